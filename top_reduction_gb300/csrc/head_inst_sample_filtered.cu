// head_inst_sample_filtered.cu -- instantiates the head kernel sampling, candidate tokens scored.
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampFiltered)
}  // namespace lmh
