// head_inst_plain_hv.cu -- instantiates the head kernel without sampling for W stored [H x V].
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampNone, true)
}  // namespace lmh
