// noalloc.cu -- lmh_logprobs_from_logits_static: the logits-chunk reduction
// for callers that cannot allocate device memory.
//
// The pages have no counterpart for this entry point; it is a convenience of
// this library.  Some callers have no way to provide a workspace:
//   * a serving engine that handed all free HBM to its KV-cache pool at
//     start-up, so nothing is left for per-step scratch;
//   * plain C host code that embeds this library without access to the
//     framework's allocator;
//   * latency-critical loops where cudaMalloc / cudaFree would synchronise
//     the device.
// This variant runs the same kernels as lmh_logprobs_from_logits (the
// logits stream and the per-row select) but keeps their intermediate results
// in a fixed array in the library's own device memory, so the call allocates
// nothing.  Its launches are recorded by the kernel trace like those of the
// workspace entry point (launch_logits_reduce brackets every launch).
//
// Limits and sharing:
//   * the array holds kStaticScratchBytes (8 MiB) on every GPU that loads
//     the library, until the process exits;
//   * requests whose partials do not fit are rejected with
//     LMH_ERR_WORKSPACE_TOO_SMALL before anything is launched (about
//     rows * (4 * ceil(V / 64) + 8 * slots + 8) bytes: up to 479 rows of
//     248320 logits, 782 rows of 151936);
//   * every call uses the same array and it keeps the previous call's
//     contents; nothing in it needs to start at zero (the chunk counter's base
//     is checked before use, and every other slot is written before it is read),
//     but calls that overlap on the GPU (two streams, or two threads) race on
//     it and must be serialised by the caller;
//   * the first call on each device does a one-time set-up with that device
//     current (kernel attributes and the array's device address through
//     cudaGetSymbolAddress); make that first call before any stream capture.
#include <mutex>

#include "lmh.h"
#include "lmh_internal.h"

namespace lmh {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(8) << 20;

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol: the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxStaticDevices];
int g_static_sms[kMaxStaticDevices];

// Once per device, with that device current: kernel attributes, SM count and
// the device address of the scratch array.
cudaError_t static_setup(void** ptr, int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = logits_reduce_setup();
    void* p = nullptr;
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_static_sms[dev] = sms;
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  *num_sms = g_static_sms[dev];
  return cudaSuccess;
}
}  // namespace

}  // namespace lmh

using namespace lmh;

extern "C" lmh_status lmh_logprobs_from_logits_static(const void* logits, lmh_dtype dtype, int32_t rows,
                                                      int32_t V, int64_t row_stride, const int32_t* sel_ids,
                                                      const int32_t* row_k, int32_t k_max, float* lse,
                                                      float* sel_logprob, int32_t* topk_ids, float* topk_logprobs,
                                                      uint32_t* dev_status, cudaStream_t stream) {
  if (rows < 0 || V <= 0 || row_stride < V) return LMH_ERR_INVALID_ARG;
  if (dtype != LMH_BF16 && dtype != LMH_F16 && dtype != LMH_F32) return LMH_ERR_INVALID_ARG;
  if (k_max < LMH_K_FULL || k_max > LMH_K_MAX) return LMH_ERR_UNSUPPORTED;
  if (k_max > V) return LMH_ERR_INVALID_ARG;
  if (!logits || !lse || (sel_ids && !sel_logprob) || (k_max > 0 && (!topk_ids || !topk_logprobs)))
    return LMH_ERR_INVALID_ARG;
  if (k_max == LMH_K_FULL && (!topk_logprobs || (reinterpret_cast<uintptr_t>(topk_logprobs) % 16) != 0))
    return LMH_ERR_INVALID_ARG;
  const int64_t elem = dtype == LMH_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(logits) % static_cast<uintptr_t>(elem)) != 0) return LMH_ERR_UNSUPPORTED;
  if (rows == 0) return LMH_OK;
  void* scratch = nullptr;
  int sms = 0;
  if (static_setup(&scratch, &sms) != cudaSuccess) return LMH_ERR_CUDA;
  const VocabSplit vs = logits_reduce_split(rows, V, k_max, sms);
  if (static_cast<int64_t>(rows) * vs.splits > INT32_MAX) return LMH_ERR_UNSUPPORTED;
  if (stream_partials_bytes(rows, vs) > kStaticScratchBytes) return LMH_ERR_WORKSPACE_TOO_SMALL;
  const Partials parts = carve_stream_partials(scratch, rows, vs);
  const cudaError_t e = launch_logits_reduce(logits, dtype, row_stride, rows, V, vs, sel_ids, row_k, k_max, parts,
                                             lse, sel_logprob, topk_ids, topk_logprobs, dev_status, stream);
  return e == cudaSuccess ? LMH_OK : LMH_ERR_CUDA;
}
