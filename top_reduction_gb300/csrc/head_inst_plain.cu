// head_inst_plain.cu -- instantiates the head kernel without sampling for W stored [V x H].
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampNone, false)
}  // namespace lmh
