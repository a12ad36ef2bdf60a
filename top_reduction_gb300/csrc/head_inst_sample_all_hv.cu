// head_inst_sample_all_hv.cu -- instantiates the head kernel with sampling, every token scored, for W stored [H x V].
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampAll, true)
}  // namespace lmh
