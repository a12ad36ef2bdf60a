// head_inst_sample_filtered.cu -- instantiates the head kernel with sampling, candidate tokens scored, for W stored [V x H].
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampFiltered, false)
}  // namespace lmh
