// head_inst_plain.cu -- instantiates the head kernel without sampling.
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampNone)
}  // namespace lmh
