// head_inst_sample_all.cu -- instantiates the head kernel sampling, every token scored.
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampAll)
}  // namespace lmh
