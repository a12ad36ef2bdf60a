// logits_reduce.cu -- standalone per-row reduction of given logits (K4).
//
// MTPLX PR #532, "Change": per row, one fp32 logsumexp; top-k ids through a
// block-max prefilter over 64-logit blocks that keeps the k blocks with the
// largest maxima, followed by an exact top-k among their entries; exact ties
// by ascending token id.
//
// GB300 design, two kernels:
//   * logits_stream_kernel -- a persistent grid (two CTAs per SM) splits the
//     flattened (row, 64-block) space of the whole chunk into equal
//     contiguous ranges, so every CTA streams the same number of bytes
//     whatever the row length.  A CTA streams its range in chunks of 2048
//     coalesced 16-byte vectors (eight per thread), issuing the next chunk's
//     loads before it works on the current one, and folds every vector into
//     the maxima of the 64-blocks (the 8 or 16 lanes of a block combine by
//     shuffles; written to the workspace) and a per-thread running max m and
//     sum exp(x - m) (online rescaling; one (m, s) per row piece after a CTA
//     reduction).  It also picks up the selected token's logit.
//   * logits_select_kernel -- one CTA per row: lse from the row pieces'
//     (m, s); tau = the k-th largest block maximum of the row (radix
//     select); candidates = entries >= tau of the blocks whose maximum is
//     >= tau, re-read from L2/HBM (the true top-k lies among them, because
//     the k blocks ranked first each hold an entry >= tau); the exact top-k
//     of the candidates by key (value desc, id asc), ordered by rank.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

constexpr int kRThreads = 256;
constexpr int kRVecPerThread = 8;  // 16-byte vectors per thread per chunk
constexpr int kRMaxPer = 4096;     // blocks per range: bounds the block-max buffer
constexpr int kRMinPer = 32;       // >= 2048 logits per range
constexpr int kRCandCap = 512;
constexpr int kRCtasPerSm = 2;

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
  __device__ __forceinline__ static float at(const void* base, int64_t i) {
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
  __device__ __forceinline__ static float at(const void* base, int64_t i) {
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
  __device__ __forceinline__ static float at(const void* base, int64_t i) {
    return reinterpret_cast<const float*>(base)[i];
  }
};

template <typename T>
__device__ __forceinline__ T neg_inf();
template <>
__device__ __forceinline__ __nv_bfloat16 neg_inf<__nv_bfloat16>() {
  return __ushort_as_bfloat16(static_cast<unsigned short>(0xFF80u));
}
template <>
__device__ __forceinline__ __half neg_inf<__half>() {
  return __ushort_as_half(static_cast<unsigned short>(0xFC00u));
}
template <>
__device__ __forceinline__ float neg_inf<float>() {
  return -INFINITY;
}

struct ReduceArgs {
  const char* logits;
  int64_t row_stride;  // elements
  int rows, V, nblk;   // nblk = 64-blocks per row
  int64_t nb_total;    // rows * nblk
  int per;             // blocks per range
  int n_ranges;
  int P;               // partial slots per row
  const int32_t* sel;
  const int32_t* row_k;
  int k_max;
  Partials parts;
  uint32_t* dev_status;
};

// One chunk of a CTA's work: up to CH blocks of one row inside one range.
struct Chunk {
  int row, lb, nbk;  // row, first block in the row, blocks
  int range;
  bool valid;
};

// Walks the chunks of the ranges blockIdx.x, blockIdx.x + gridDim.x, ...
// (row and block advance incrementally; one division per range).
template <int CH>
struct ChunkIter {
  int64_t left;  // blocks left in the current range
  int row, lb, range;
  bool done;
  __device__ void start(const ReduceArgs& a) {
    if (range >= a.n_ranges) {
      done = true;
      return;
    }
    const int64_t b = static_cast<int64_t>(range) * a.per;
    left = min(static_cast<int64_t>(a.per), a.nb_total - b);
    row = static_cast<int>(b / a.nblk);
    lb = static_cast<int>(b - static_cast<int64_t>(row) * a.nblk);
  }
  __device__ void init(const ReduceArgs& a) {
    range = blockIdx.x;
    done = false;
    start(a);
  }
  __device__ Chunk next(const ReduceArgs& a) {
    Chunk c;
    c.valid = false;
    c.row = c.lb = c.nbk = c.range = 0;
    if (done) return c;
    if (left == 0) {
      range += gridDim.x;
      start(a);
      if (done) return c;
    }
    c.row = row;
    c.lb = lb;
    c.nbk = static_cast<int>(min(static_cast<int64_t>(CH), min(left, static_cast<int64_t>(a.nblk - lb))));
    c.range = range;
    c.valid = true;
    left -= c.nbk;
    lb += c.nbk;
    if (lb == a.nblk) {
      lb = 0;
      ++row;
    }
    return c;
  }
};

// The chunk's vectors v = threadIdx.x + j * kRThreads (j < kRVecPerThread)
// held in registers; `ne` logits of the chunk are real, the rest read as -inf.
template <typename T>
struct ChunkRegs {
  uint4 w[kRVecPerThread];
  int ne;

  __device__ __forceinline__ void load(const ReduceArgs& a, const Chunk& c) {
    constexpr int EPV = Vec16<T>::N;
    const T* src = reinterpret_cast<const T*>(a.logits) + static_cast<int64_t>(c.row) * a.row_stride +
                   static_cast<int64_t>(c.lb) * kBlock;
    ne = min(c.nbk * kBlock, a.V - c.lb * kBlock);
    const bool vec_ok = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
#pragma unroll
    for (int j = 0; j < kRVecPerThread; ++j) {
      const int v = threadIdx.x + j * kRThreads;
      const int first = v * EPV;
      if (vec_ok && first + EPV <= ne) {
        w[j] = __ldcs(reinterpret_cast<const uint4*>(src) + v);  // streamed once: evict-first
      } else {
        // ragged tail or unaligned row: element loads, -inf beyond the row
        alignas(16) T t[EPV];
#pragma unroll
        for (int e = 0; e < EPV; ++e) t[e] = (first + e < ne) ? src[first + e] : neg_inf<T>();
        w[j] = *reinterpret_cast<uint4*>(t);
      }
    }
  }
};

template <typename T>
__global__ void __launch_bounds__(kRThreads, kRCtasPerSm) logits_stream_kernel(const ReduceArgs a) {
  using VT = Vec16<T>;
  constexpr int EPV = VT::N;                                        // elements per 16-byte vector
  constexpr int VPB = kBlock / EPV;                                 // vectors per 64-block
  constexpr int CH = kRVecPerThread * kRThreads / VPB;              // blocks per chunk
  constexpr int kValueBits = VT::kKeyBits;
  constexpr uint32_t kMask = kValueBits >= 32 ? 0xFFFFFFFFu : (0xFFFFFFFFu << (32 - kValueBits));

  __shared__ float red[32];
  pdl_launch_dependents();  // the select kernel may be scheduled now; it waits for this grid's results

  ChunkIter<CH> it;
  it.init(a);
  Chunk cur = it.next(a);
  ChunkRegs<T> buf0, buf1;  // two register buffers with fixed roles per half of the unrolled loop
  if (cur.valid) buf0.load(a, cur);

  const float L = kLog2e;
  float tm = -INFINITY, ts = 0.0f;  // this thread's running max / sum over the current piece
  int piece_blocks = 0, sel_rel = -1;
  auto step = [&](ChunkRegs<T>& cb, ChunkRegs<T>& nb) {
    const Chunk nxt = it.next(a);
    if (nxt.valid) nb.load(a, nxt);  // in flight while this chunk is worked on
    if (piece_blocks == 0) sel_rel = a.sel ? a.sel[cur.row] : -1;
    const int ne = cb.ne;
    const int rel0 = sel_rel - cur.lb * kBlock;  // selected token relative to this chunk

    // ---- block maxima + online (m, s) ----
#pragma unroll
    for (int j = 0; j < kRVecPerThread; ++j) {
      const int v = threadIdx.x + j * kRThreads;
      float x[EPV];
      VT::load(&cb.w[j], x);
      float vm = x[0];
#pragma unroll
      for (int e = 1; e < EPV; ++e) vm = fmaxf(vm, x[e]);
      if (vm > tm) {
        ts = (tm == -INFINITY) ? 0.0f : ts * ex2_approx((tm - vm) * L);
        tm = vm;
      }
      if (tm != -INFINITY) {
        const float mL = tm * L;
#pragma unroll
        for (int e = 0; e < EPV; ++e) ts += ex2_approx(fmaf(x[e], L, -mL));
      }
      const unsigned r = static_cast<unsigned>(rel0 - v * EPV);
      if (r < static_cast<unsigned>(EPV) && rel0 < ne) {  // the token is one of this chunk's real logits
        float sv = 0.0f;
#pragma unroll
        for (int e = 0; e < EPV; ++e) sv = (static_cast<unsigned>(e) == r) ? x[e] : sv;
        a.parts.sel_logit[cur.row] = sv;
      }
#pragma unroll
      for (int o = VPB / 2; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
      if (v * EPV < cur.nbk * kBlock && (threadIdx.x % VPB) == 0)
        a.parts.bmax[static_cast<int64_t>(cur.row) * a.nblk + cur.lb + v / VPB] = vm;
    }
    piece_blocks += cur.nbk;

    const bool piece_end = !nxt.valid || nxt.row != cur.row || nxt.range != cur.range;
    if (piece_end) {
      const int row = cur.row;
      const int slot = cur.range - static_cast<int>((static_cast<int64_t>(row) * a.nblk) / a.per);
      const float M = block_max(tm, red);
      const float S = block_sum((tm == -INFINITY) ? 0.0f : ts * expf(tm - M), red);
      if (threadIdx.x == 0) a.parts.part_ms[static_cast<int64_t>(row) * a.P + slot] = make_float2(M, M == -INFINITY ? 0.0f : S);
      tm = -INFINITY;
      ts = 0.0f;
      piece_blocks = 0;
    }
    cur = nxt;
  };
  while (cur.valid) {
    step(buf0, buf1);
    if (!cur.valid) break;
    step(buf1, buf0);
  }
}

// ---------------------------------------------------------------------------
// per-row selection
// ---------------------------------------------------------------------------
constexpr int kSThreads = 256;
constexpr int kSKeptCap = 1024;  // kept blocks held in shared memory
constexpr int kSCandCap = 512;   // candidate keys held in shared memory
constexpr int kSStageBlocks = 16384;  // block maxima staged in shared memory (V <= 1,048,576)

template <typename T>
__global__ void __launch_bounds__(kSThreads) logits_select_kernel(const ReduceArgs a, float* lse_out,
                                                                  float* sel_logprob, int32_t* topk_ids,
                                                                  float* topk_logprobs) {
  using VT = Vec16<T>;
  constexpr int kValueBits = VT::kKeyBits;
  constexpr uint32_t kMask = kValueBits >= 32 ? 0xFFFFFFFFu : (0xFFFFFFFFu << (32 - kValueBits));
  __shared__ uint64_t cand[kSCandCap];
  __shared__ int kept[kSKeptCap];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t misc[4];  // [0] candidates, [1..2] select broadcast, [3] kept blocks
  __shared__ float red[32];
  pdl_wait();  // the block maxima and (m, s) come from the stream kernel just before

  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  // ---- lse over the row's pieces ----
  const int64_t b0 = static_cast<int64_t>(row) * a.nblk;
  const int nslots = static_cast<int>((b0 + a.nblk - 1) / a.per - b0 / a.per) + 1;
  const float2* ms = a.parts.part_ms + static_cast<int64_t>(row) * a.P;
  float tm = -INFINITY, ts = 0.0f;
  for (int j = tid; j < nslots; j += kSThreads) {
    const float2 p = ms[j];
    if (p.x > tm) {
      ts = (tm == -INFINITY) ? 0.0f : ts * expf(tm - p.x);
      tm = p.x;
    }
    if (p.x != -INFINITY) ts += p.y * expf(p.x - tm);
  }
  const float M = block_max(tm, red);
  const float S = block_sum((tm == -INFINITY) ? 0.0f : ts * expf(tm - M), red);
  const float lse = (M == -INFINITY) ? -INFINITY : M + logf(S);
  if (tid == 0) {
    lse_out[row] = lse;
    if (a.sel) {
      const int t = a.sel[row];
      float v = __int_as_float(0x7fc00000);  // NaN: no selected token / out of range
      if (t >= 0 && t < a.V)
        v = a.parts.sel_logit[row] - lse;
      else if (t != -1)
        set_status(a.dev_status, LMH_DS_SEL_OUT_OF_RANGE);
      sel_logprob[row] = v;
    }
    misc[0] = 0;
    misc[3] = 0;
  }
  if (a.k_max == 0) return;
  int k = a.k_max;
  if (a.row_k) k = min(max(a.row_k[row], 0), a.k_max);
  int32_t* out_ids = topk_ids + static_cast<int64_t>(row) * a.k_max;
  float* out_lp = topk_logprobs + static_cast<int64_t>(row) * a.k_max;
  if (k == 0) {
    for (int r = tid; r < a.k_max; r += kSThreads) {
      out_ids[r] = -1;
      out_lp[r] = -INFINITY;
    }
    return;
  }

  // ---- tau: the k-th largest block maximum of the row ----
  // The row's block maxima are staged in shared memory (one coalesced round)
  // when they fit; otherwise they are read from global memory (L2).
  extern __shared__ float sbm[];
  const int nb = a.nblk;
  const float* bm = a.parts.bmax + b0;
  if (nb <= kSStageBlocks) {
    for (int b = tid; b < nb; b += kSThreads) sbm[b] = bm[b];
    __syncthreads();
    bm = sbm;
  }
  uint32_t thr = 0;  // ord(tau) restricted to the top kValueBits bits; 0 keeps every entry
  if (nb > k) {
    int above;
    const uint64_t T64 = cta_radix_select(
        [&](int b, uint64_t* key) {
          *key = static_cast<uint64_t>(f32_ord(bm[b])) << 32;
          return true;
        },
        nb, k, kValueBits, hist, misc + 1, &above);
    thr = static_cast<uint32_t>(T64 >> 32);
  }
  __syncthreads();
  // ---- kept blocks (order is irrelevant: candidates are ranked below) ----
  for (int b = tid; b < nb; b += kSThreads)
    if ((f32_ord(bm[b]) & kMask) >= thr) {
      const uint32_t pos = atomicAdd(&misc[3], 1u);
      if (pos < kSKeptCap) kept[pos] = b;
    }
  __syncthreads();
  const int nkept = static_cast<int>(misc[3]);
  const T* rowp = reinterpret_cast<const T*>(a.logits) + static_cast<int64_t>(row) * a.row_stride;
  auto in_set = [&](int i, uint64_t* key) -> bool {  // i over the whole row (fallback)
    if ((f32_ord(bm[i / kBlock]) & kMask) < thr || i >= a.V) return false;
    const float x = VT::at(rowp, i);
    if ((f32_ord(x) & kMask) < thr) return false;
    *key = make_key(x, i);
    return true;
  };
  int cnt;
  if (nkept <= kSKeptCap) {
    // gather the kept blocks' entries >= tau: every load of the CTA in one round
    const int n_el = nkept * kBlock;
    for (int i = tid; i < n_el; i += kSThreads) {
      const int e = kept[i / kBlock] * kBlock + (i % kBlock);
      if (e >= a.V) continue;
      const float x = VT::at(rowp, e);
      if ((f32_ord(x) & kMask) < thr) continue;
      const uint32_t pos = atomicAdd(&misc[0], 1u);
      if (pos < kSCandCap) cand[pos] = make_key(x, e);
    }
    __syncthreads();
    cnt = static_cast<int>(misc[0]);
  } else {
    cnt = kSCandCap + 1;  // too many ties at tau for the lists: take the exact path
  }
  if (cnt > kSCandCap) {
    int above;
    const int n_items = nb * kBlock;
    const uint64_t T64 = cta_radix_select(in_set, n_items, k, 64, hist, misc + 1, &above);
    __syncthreads();
    if (tid == 0) misc[0] = 0;
    __syncthreads();
    for (int i = tid; i < n_items; i += kSThreads) {
      uint64_t key = 0;
      if (in_set(i, &key) && key >= T64) {
        const uint32_t pos = atomicAdd(&misc[0], 1u);  // exactly k of them
        if (pos < kSCandCap) cand[pos] = key;
      }
    }
    __syncthreads();
    cnt = min(k, static_cast<int>(misc[0]));
  }
  // ---- exact order by rank (keys are unique) ----
  for (int t = tid; t < cnt; t += kSThreads) {
    const uint64_t key = cand[t];
    int rank = 0;
    for (int j = 0; j < cnt; ++j) rank += cand[j] > key;
    if (rank < k) {
      out_ids[rank] = key_id(key);
      out_lp[rank] = key_value(key) - lse;
    }
  }
  for (int r = min(cnt, k) + tid; r < a.k_max; r += kSThreads) {  // ranks without a candidate, and ranks >= k
    out_ids[r] = -1;
    out_lp[r] = -INFINITY;
  }
}

VocabSplit logits_reduce_split(int rows, int V, int k_max, int num_sms) {
  VocabSplit vs;
  const int nblk = (V + kBlock - 1) / kBlock;
  const int64_t nb_total = static_cast<int64_t>(rows) * nblk;
  const int64_t G = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * kRCtasPerSm;
  int64_t per = (nb_total + G - 1) / G;
  // a range of more than 2k blocks lets the block-max threshold prune (<= k blocks keep everything)
  const int64_t min_per = 2 * k_max > kRMinPer ? 2 * k_max : kRMinPer;
  if (per < min_per) per = min_per;
  if (per > kRMaxPer) per = kRMaxPer;
  vs.per = static_cast<int>(per);
  vs.n_ranges = static_cast<int>((nb_total + per - 1) / per);
  vs.grid = static_cast<int>(vs.n_ranges < G ? vs.n_ranges : G);
  vs.splits = static_cast<int>((nblk + per - 1) / per) + 1;  // row pieces per row, at most
  vs.nblk = nblk;
  return vs;
}

cudaError_t logits_reduce_setup() {
  const int bytes = kSStageBlocks * static_cast<int>(sizeof(float));
  cudaError_t e =
      cudaFuncSetAttribute(logits_select_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(logits_select_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(logits_select_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

size_t stream_partials_bytes(int rows, const VocabSplit& vs) {
  auto al = [](size_t n) { return (n + 255) & ~static_cast<size_t>(255); };
  return al(static_cast<size_t>(rows) * vs.splits * 8) + al(static_cast<size_t>(rows) * 4) +
         al(static_cast<size_t>(rows) * vs.nblk * 4);
}

Partials carve_stream_partials(void* base, int rows, const VocabSplit& vs) {
  auto al = [](size_t n) { return (n + 255) & ~static_cast<size_t>(255); };
  char* p = static_cast<char*>(base);
  Partials out;
  out.part_ms = reinterpret_cast<float2*>(p);
  p += al(static_cast<size_t>(rows) * vs.splits * 8);
  out.sel_logit = reinterpret_cast<float*>(p);
  p += al(static_cast<size_t>(rows) * 4);
  out.bmax = reinterpret_cast<float*>(p);
  out.part_keys = nullptr;
  return out;
}

template <typename T>
static cudaError_t launch_both(const ReduceArgs& a, const VocabSplit& split, float* lse, float* sel_logprob,
                               int32_t* topk_ids, float* topk_logprobs, cudaStream_t stream, TraceKernel tk_select) {
  cudaError_t e;
  {
    trace_begin(kTraceReduce, stream);
    e = launch_kernel(logits_stream_kernel<T>, dim3(split.grid), dim3(kRThreads), 0, stream, false, a);
    trace_end(kTraceReduce, stream);
  }
  if (e != cudaSuccess) return e;
  trace_begin(tk_select, stream);
  const size_t smem = static_cast<size_t>(min(a.nblk, kSStageBlocks)) * sizeof(float);
  e = launch_kernel(logits_select_kernel<T>, dim3(a.rows), dim3(kSThreads), smem, stream, true, a, lse, sel_logprob,
                    topk_ids, topk_logprobs);
  trace_end(tk_select, stream);
  return e;
}

cudaError_t launch_logits_reduce(const void* logits, lmh_dtype dtype, int64_t row_stride, int rows, int V,
                                 VocabSplit split, const int32_t* sel, const int32_t* row_k, int k_max,
                                 Partials parts, float* lse, float* sel_logprob, int32_t* topk_ids,
                                 float* topk_logprobs, uint32_t* dev_status, cudaStream_t stream) {
  ReduceArgs a;
  a.logits = static_cast<const char*>(logits);
  a.row_stride = row_stride;
  a.rows = rows;
  a.V = V;
  a.nblk = split.nblk;
  a.nb_total = static_cast<int64_t>(rows) * split.nblk;
  a.per = split.per;
  a.n_ranges = split.n_ranges;
  a.P = split.splits;
  a.sel = sel;
  a.row_k = row_k;
  a.k_max = k_max;
  a.parts = parts;
  a.dev_status = dev_status;
  switch (dtype) {
    case LMH_BF16:
      return launch_both<__nv_bfloat16>(a, split, lse, sel_logprob, topk_ids, topk_logprobs, stream, kTraceLogitsSelect);
    case LMH_F16:
      return launch_both<__half>(a, split, lse, sel_logprob, topk_ids, topk_logprobs, stream, kTraceLogitsSelect);
    default:
      return launch_both<float>(a, split, lse, sel_logprob, topk_ids, topk_logprobs, stream, kTraceLogitsSelect);
  }
}

}  // namespace lmh
