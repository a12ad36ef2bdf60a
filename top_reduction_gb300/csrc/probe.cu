// probe.cu -- element comparison for lmh_probe_selective.
//
// vllm-metal release v0.4.0.dev20260831, "Summary": the selective head is
// used only when it reproduces the model's own output (bit-exact there); an
// engine keeps full logits otherwise.  This kernel counts the elements of two
// f32 arrays that differ by more than a tolerance.
#include <cmath>

#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

// Grid-stride over n elements; one atomic per warp and pass.
__global__ void __launch_bounds__(256) probe_compare_kernel(const float* __restrict__ ours,
                                                            const float* __restrict__ ref, int64_t n, float tol,
                                                            uint32_t* count) {
  pdl_wait();  // the head kernel that wrote `ours` may still be finishing
  const int lane = threadIdx.x & 31;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < n; base += stride) {
    const int64_t i = base + threadIdx.x;
    bool bad = false;
    if (i < n) {
      const float a = ours[i], b = ref[i];
      const bool na = isnan(a), nb = isnan(b);
      bad = (na != nb) || (!na && !(fabsf(a - b) <= tol) && a != b);
    }
    const unsigned m = __ballot_sync(0xffffffffu, bad);
    if (lane == 0 && m) atomicAdd(count, static_cast<uint32_t>(__popc(m)));
  }
}

cudaError_t launch_probe_compare(const float* ours, const float* ref, int64_t n, float tol, uint32_t* count,
                                 int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess || n == 0) return e;
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  return launch_kernel(probe_compare_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, false, ours,
                       ref, n, tol, count);
}

}  // namespace lmh
