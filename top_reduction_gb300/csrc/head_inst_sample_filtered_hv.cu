// head_inst_sample_filtered_hv.cu -- instantiates the head kernel with sampling, candidate tokens scored, for W stored [H x V].
#include "head_kernel.cuh"

namespace lmh {
LMH_HEAD_MODE_DECL(, kSampFiltered, true)
}  // namespace lmh
