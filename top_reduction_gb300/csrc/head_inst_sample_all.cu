// head_inst_sample_all.cu -- instantiates the head kernel with sampling, every token scored, for W stored [V x H].
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampAll, false)
}  // namespace lmh
