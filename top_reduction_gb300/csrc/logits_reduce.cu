// logits_reduce.cu -- standalone per-row reduction of given logits (K4).
//
// MTPLX PR #532, "Change": per row, one fp32 logsumexp; top-k ids through a
// block-max prefilter over 64-logit blocks that keeps the k blocks with the
// largest maxima, followed by an exact top-k among their entries; exact ties
// by ascending token id.
//
// GB300 design: one CTA per (row, chunk) where a chunk is a run of whole
// 64-blocks of the row.  A single bulk copy (TMA engine) brings the chunk into
// shared memory; the CTA then makes its passes there:
//   A. block maxima (16-byte vectors, the 8 or 16 lanes of a block combine
//      with shuffles) and the chunk maximum m;
//   B. s = sum exp(x - m) with ex2 on the SFU;
//   C. the k-th largest block maximum tau (radix select on the block maxima);
//   D. candidates = entries >= tau inside blocks whose max >= tau (the true
//      top-k of the chunk lies among them: the k kept blocks each hold an
//      entry >= tau), then an exact top-k of the candidates by key.
// The chunk's (m, s), its sorted top-k keys and, if the chunk holds it, the
// selected token's logit go to the workspace; merge_partials.cu combines the
// chunks of a row.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

constexpr int kReduceThreads = 256;
constexpr int kReduceCandCap = 512;  // candidate keys held in shared memory
constexpr int kReduceMaxBlocksPerSplit = 256;

template <typename T>
struct Vec16;  // 16-byte vector of T widened to fp32

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static constexpr int kKeyBits = 16;  // a bf16 value is exact in the top 16 bits of its fp32 key
  __device__ __forceinline__ static void load(const void* p, float* x) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(u[i] << 16);
      x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static float at(const void* base, int i) {
    const uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
};

template <>
struct Vec16<__half> {
  static constexpr int N = 8;
  static constexpr int kKeyBits = 32;
  __device__ __forceinline__ static void load(const void* p, float* x) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static float at(const void* base, int i) {
    return __half2float(reinterpret_cast<const __half*>(base)[i]);
  }
};

template <>
struct Vec16<float> {
  static constexpr int N = 4;
  static constexpr int kKeyBits = 32;
  __device__ __forceinline__ static void load(const void* p, float* x) {
    const float4 w = *reinterpret_cast<const float4*>(p);
    x[0] = w.x;
    x[1] = w.y;
    x[2] = w.z;
    x[3] = w.w;
  }
  __device__ __forceinline__ static float at(const void* base, int i) {
    return reinterpret_cast<const float*>(base)[i];
  }
};

struct ReduceArgs {
  const char* logits;
  int64_t row_stride;  // elements
  int rows, V, splits, bps;
  const int32_t* sel;
  const int32_t* row_k;
  int k_max;
  Partials parts;
  uint32_t* dev_status;
};

template <typename T>
__global__ void __launch_bounds__(kReduceThreads) logits_reduce_kernel(const ReduceArgs a) {
  using VT = Vec16<T>;
  constexpr int EPV = VT::N;                // elements per 16-byte vector
  constexpr int VPB = kBlock / EPV;         // vectors per 64-block
  constexpr int kValueBits = VT::kKeyBits;  // key bits that order the values exactly

  extern __shared__ __align__(128) unsigned char smem[];
  const int row = blockIdx.x / a.splits;
  const int split = blockIdx.x % a.splits;
  const int nblk_row = (a.V + kBlock - 1) / kBlock;
  const int b0 = split * a.bps;
  const int nb = min(a.bps, nblk_row - b0);
  const int e0 = b0 * kBlock;
  const int ne = min(nb * kBlock, a.V - e0);

  // shared layout: chunk | bmax[bps] | cand[cap] | hist[256] | misc[4] | red[32] | barrier
  const int chunk_bytes = ((a.bps * kBlock * static_cast<int>(sizeof(T))) + 15) & ~15;
  T* chunk = reinterpret_cast<T*>(smem);
  float* bmax = reinterpret_cast<float*>(smem + chunk_bytes);
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem + chunk_bytes + ((a.bps * 4 + 15) & ~15));
  uint32_t* hist = reinterpret_cast<uint32_t*>(cand + kReduceCandCap);
  uint32_t* misc = hist + 256;                            // [0] candidate count, [1..2] select broadcast
  float* red = reinterpret_cast<float*>(misc + 4);        // 32 floats
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + 32);  // 16-byte aligned offset

  const char* src =
      a.logits + (static_cast<int64_t>(row) * a.row_stride + e0) * static_cast<int64_t>(sizeof(T));
  const uint32_t bytes = static_cast<uint32_t>(ne) * sizeof(T);
  const uint32_t bulk = bytes & ~15u;

  // rows whose start is 16-byte aligned arrive by one bulk copy; any other
  // row pitch is copied by the whole CTA with plain element loads
  const bool use_bulk = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init_fence();
    misc[0] = 0;
  }
  __syncthreads();
  if (use_bulk) {
    if (threadIdx.x == 0) {
      if (bulk > 0) {
        mbar_arrive_expect_tx(bar, bulk);
        bulk_load(chunk, src, bulk, bar);
      } else {
        mbar_arrive(bar);
      }
      // ragged tail (< 16 bytes) with plain loads
      for (uint32_t o = bulk; o < bytes; o += sizeof(T))
        *reinterpret_cast<T*>(reinterpret_cast<char*>(chunk) + o) = *reinterpret_cast<const T*>(src + o);
    }
  } else {
    if (threadIdx.x == 0) mbar_arrive(bar);
    const T* s = reinterpret_cast<const T*>(src);
    for (int i = threadIdx.x; i < ne; i += kReduceThreads) chunk[i] = s[i];
  }
  const bool ok = mbar_wait(bar, 0);
  if (!ok) {
    if (threadIdx.x == 0) set_status(a.dev_status, LMH_DS_TIMEOUT);
    return;
  }
  __syncthreads();  // the plain-load parts

  // ---- pass A: block maxima and the chunk maximum ----
  const int nvec = nb * VPB;
  float tmax = -INFINITY;
  for (int base = 0; base < nvec; base += kReduceThreads) {
    const int v = base + threadIdx.x;
    float x[EPV];
    float vm = -INFINITY;
    if (v < nvec) {
      VT::load(reinterpret_cast<const char*>(chunk) + v * 16, x);
      const int first = v * EPV;
      if (first + EPV <= ne) {
#pragma unroll
        for (int j = 0; j < EPV; ++j) vm = fmaxf(vm, x[j]);
      } else {
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if (first + j < ne) vm = fmaxf(vm, x[j]);
      }
    }
    tmax = fmaxf(tmax, vm);
#pragma unroll
    for (int o = VPB / 2; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
    if (v < nvec && (threadIdx.x % VPB) == 0) bmax[v / VPB] = vm;
  }
  const float m = block_max(tmax, red);

  // ---- pass B: s = sum exp(x - m) ----
  float tsum = 0.0f;
  if (m != -INFINITY) {
    const float mL = m * kLog2e;
    for (int v = threadIdx.x; v < nvec; v += kReduceThreads) {
      float x[EPV];
      VT::load(reinterpret_cast<const char*>(chunk) + v * 16, x);
      const int first = v * EPV;
      if (first + EPV <= ne) {
#pragma unroll
        for (int j = 0; j < EPV; ++j) tsum += ex2_approx(fmaf(x[j], kLog2e, -mL));
      } else {
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if (first + j < ne) tsum += ex2_approx(fmaf(x[j], kLog2e, -mL));
      }
    }
  }
  const float s = block_sum(tsum, red);

  const int64_t pidx = static_cast<int64_t>(row) * a.splits + split;
  if (threadIdx.x == 0) {
    a.parts.part_ms[pidx] = make_float2(m, s);
    const int t = a.sel ? a.sel[row] : -1;
    if (t >= e0 && t < e0 + ne) a.parts.sel_logit[row] = VT::at(chunk, t - e0);
  }

  int k = a.k_max;
  if (a.row_k) k = min(max(a.row_k[row], 0), a.k_max);
  if (k == 0) return;

  // ---- pass C: tau = the k-th largest block maximum ----
  uint32_t thr = 0;  // ord(tau) restricted to the top kValueBits bits; 0 keeps every entry
  constexpr uint32_t kMask = kValueBits >= 32 ? 0xFFFFFFFFu : (0xFFFFFFFFu << (32 - kValueBits));
  if (nb > k) {
    int above;
    const uint64_t T64 = cta_radix_select(
        [&](int i, uint64_t* key) {
          *key = static_cast<uint64_t>(f32_ord(bmax[i])) << 32;
          return true;
        },
        nb, k, kValueBits, hist, misc + 1, &above);
    thr = static_cast<uint32_t>(T64 >> 32);
  }

  // ---- pass D: candidates, then the exact top-k among them ----
  auto in_set = [&](int i, uint64_t* key) -> bool {
    const int b = i / kBlock;
    if ((f32_ord(bmax[b]) & kMask) < thr) return false;
    if (i >= ne) return false;
    const float x = VT::at(chunk, i);
    if ((f32_ord(x) & kMask) < thr) return false;
    *key = make_key(x, e0 + i);
    return true;
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = warp; b < nb; b += kReduceThreads / 32) {
    if ((f32_ord(bmax[b]) & kMask) < thr) continue;  // warp-uniform: block pruned
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = b * kBlock + h * 32 + lane;
      uint64_t key = 0;
      const bool in = in_set(i, &key);
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      uint32_t basepos = 0;
      if (lane == 0 && bal) basepos = atomicAdd(&misc[0], __popc(bal));
      basepos = __shfl_sync(0xffffffffu, basepos, 0);
      if (in) {
        const uint32_t pos = basepos + __popc(bal & ((1u << lane) - 1u));
        if (pos < kReduceCandCap) cand[pos] = key;
      }
    }
  }
  __syncthreads();
  const int cnt = static_cast<int>(misc[0]);
  int nsort = cnt;
  if (cnt > kReduceCandCap) {
    // many exact ties at tau: exact radix select over the whole candidate set
    int above;
    const uint64_t T64 = cta_radix_select(in_set, nb * kBlock, k, 64, hist, misc + 1, &above);
    __syncthreads();
    if (threadIdx.x == 0) misc[0] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < nb * kBlock; i += kReduceThreads) {
      uint64_t key = 0;
      if (in_set(i, &key) && key >= T64) {
        const uint32_t pos = atomicAdd(&misc[0], 1u);  // exactly k of them
        if (pos < kReduceCandCap) cand[pos] = key;
      }
    }
    __syncthreads();
    nsort = min(k, static_cast<int>(misc[0]));
  }
  const int n2 = next_pow2(nsort);
  for (int i = nsort + threadIdx.x; i < n2; i += kReduceThreads) cand[i] = 0ull;
  cta_bitonic_sort_desc(cand, n2);
  unsigned long long* out = a.parts.part_keys + pidx * a.k_max;
  for (int j = threadIdx.x; j < k; j += kReduceThreads) out[j] = (j < nsort) ? cand[j] : 0ull;
}

VocabSplit logits_reduce_split(int rows, int V, int num_sms) {
  const int nblk = (V + kBlock - 1) / kBlock;
  const int lo = (nblk + kReduceMaxBlocksPerSplit - 1) / kReduceMaxBlocksPerSplit;  // shared-memory bound
  const int want = (4 * num_sms + rows - 1) / (rows > 0 ? rows : 1);                // enough CTAs
  const int hi = nblk / 16 > lo ? nblk / 16 : lo;                                   // >= 1024 logits each
  int splits = want < lo ? lo : (want > hi ? hi : want);
  if (splits < 1) splits = 1;
  const int bps = (nblk + splits - 1) / splits;
  VocabSplit vs;
  vs.blocks_per_split = bps;
  vs.splits = (nblk + bps - 1) / bps;
  return vs;
}

static size_t reduce_smem_bytes(int bps, int elem) {
  size_t chunk = ((static_cast<size_t>(bps) * kBlock * elem) + 15) & ~static_cast<size_t>(15);
  size_t b = ((static_cast<size_t>(bps) * 4) + 15) & ~static_cast<size_t>(15);
  return chunk + b + kReduceCandCap * 8 + 256 * 4 + 4 * 4 + 32 * 4 + 16;
}

cudaError_t logits_reduce_setup() {
  const int max2 = static_cast<int>(reduce_smem_bytes(kReduceMaxBlocksPerSplit, 2));
  const int max4 = static_cast<int>(reduce_smem_bytes(kReduceMaxBlocksPerSplit, 4));
  cudaError_t e = cudaFuncSetAttribute(logits_reduce_kernel<__nv_bfloat16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, max2);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(logits_reduce_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, max2);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(logits_reduce_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, max4);
  return e;
}

cudaError_t launch_logits_reduce(const void* logits, lmh_dtype dtype, int64_t row_stride, int rows, int V,
                                 VocabSplit split, const int32_t* sel, const int32_t* row_k, int k_max,
                                 Partials parts, uint32_t* dev_status, cudaStream_t stream) {
  ReduceArgs a;
  a.logits = static_cast<const char*>(logits);
  a.row_stride = row_stride;
  a.rows = rows;
  a.V = V;
  a.splits = split.splits;
  a.bps = split.blocks_per_split;
  a.sel = sel;
  a.row_k = row_k;
  a.k_max = k_max;
  a.parts = parts;
  a.dev_status = dev_status;
  const dim3 grid(static_cast<unsigned>(rows) * static_cast<unsigned>(split.splits));
  switch (dtype) {
    case LMH_BF16:
      logits_reduce_kernel<__nv_bfloat16><<<grid, kReduceThreads, reduce_smem_bytes(a.bps, 2), stream>>>(a);
      break;
    case LMH_F16:
      logits_reduce_kernel<__half><<<grid, kReduceThreads, reduce_smem_bytes(a.bps, 2), stream>>>(a);
      break;
    default:
      logits_reduce_kernel<float><<<grid, kReduceThreads, reduce_smem_bytes(a.bps, 4), stream>>>(a);
      break;
  }
  return cudaGetLastError();
}

}  // namespace lmh
