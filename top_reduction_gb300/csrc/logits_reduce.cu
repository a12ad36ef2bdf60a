// logits_reduce.cu -- standalone per-row reduction of given logits (K4).
//
// MTPLX PR #532, "Change": per row, one fp32 logsumexp; top-k ids through a
// block-max prefilter over 64-logit blocks that keeps the k blocks with the
// largest maxima, followed by an exact top-k among their entries; exact ties
// by ascending token id.
//
// GB300 design:
//   * a stream kernel reads every logit once, as a persistent grid over the
//     whole chunk, so the work per CTA does not depend on the row length.
//     For every 64-block it writes the block's maximum to the workspace, and
//     it folds the logits into (max m, sum exp(x - m)) pairs.  It also picks
//     up the selected token's logit.
//       - logits_stream_tma_kernel (rows and the row length 16-byte
//         aligned; four CTAs per SM): the logits are cut into 16 KB chunks
//         of one row, handed out dynamically (a ticket counter whose base the
//         previous call's select kernel recorded), so CTAs that get more
//         bandwidth take more chunks.  One producer lane streams its chunks into a ring of
//         shared-memory stages with bulk copies (cp.async.bulk, completion on
//         mbarriers); four consumer warps read them, each thread owning 128
//         contiguous bytes (one bf16/f16 block, half an f32 block), so a
//         block's maximum needs no exchange between lanes; one (m, s) pair
//         per warp and chunk.  A CTA's first three chunks are fixed and go
//         out before the grid-dependency wait, so in a sequence of calls they
//         stream while the previous call's select kernel runs.
//       - logits_stream_regs_kernel (any element-aligned layout; two CTAs
//         per SM): the flattened (row, 64-block) space is cut into equal
//         contiguous ranges, one per CTA; every thread loads 16-byte vectors
//         (or elements at unaligned rows) straight into registers, two
//         chunks in flight; the lanes of a block combine their maxima by
//         shuffles; one (m, s) pair per row piece.
//   * logits_select_kernel, one CTA per row, after the stream kernel
//     (select_row): lse from the row's (m, s) pairs (one warp); a lower bound
//     t on the row's k-th largest logit from the block maxima; candidates =
//     entries >= t of the blocks whose maximum is >= t, re-read from memory
//     with their 16-byte loads spread evenly over the CTA (one round trip);
//     their exact top-k by key (value desc, id asc), ordered by rank.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

// register-path stream kernel
constexpr int kRThreads = 256;
constexpr int kRVecPerThread = 8;  // 16-byte vectors per thread per chunk
constexpr int kRCtasPerSm = 2;
// ranges
constexpr int kRMaxPer = 4096;  // blocks per range, at most
constexpr int kRMinPer = 32;    // >= 2048 logits per range
// TMA-path stream kernel
constexpr int kTConsumerWarps = 4;
constexpr int kTConsumers = kTConsumerWarps * 32;
constexpr int kTThreads = kTConsumers + 32;  // + one producer warp
constexpr int kTChunkBytes = kTConsumers * 128;  // 128 contiguous bytes per consumer thread
constexpr int kTStages = 3;
constexpr int kTCtasPerSm = 4;
constexpr int kTDescBytes = 32;
constexpr int kTSmemRing = kTStages * kTChunkBytes + kTStages * kTDescBytes + 2 * kTStages * 8 + 16;

template <typename T>
struct Vec16;  // 16-byte vector of T widened to fp32

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;  // two bf16 -inf
  __device__ __forceinline__ static void load(const void* p, float* x) { unpack(*reinterpret_cast<const uint4*>(p), x); }
  __device__ __forceinline__ static void unpack(const uint4 w, float* x) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(u[i] << 16);
      x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  }
  // maximum of 8 vectors, pairwise on packed bf16x2 (exact)
  __device__ __forceinline__ static float max8(const uint4* w) {
    __nv_bfloat162 m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t* a = reinterpret_cast<const uint32_t*>(&w[2 * i]);
      const uint32_t* b = reinterpret_cast<const uint32_t*>(&w[2 * i + 1]);
      __nv_bfloat162 t0 = __hmax2(as2(a[0]), as2(a[1])), t1 = __hmax2(as2(a[2]), as2(a[3]));
      __nv_bfloat162 t2 = __hmax2(as2(b[0]), as2(b[1])), t3 = __hmax2(as2(b[2]), as2(b[3]));
      m[i] = __hmax2(__hmax2(t0, t1), __hmax2(t2, t3));
    }
    const __nv_bfloat162 r = __hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3]));
    return fmaxf(__low2float(r), __high2float(r));
  }
  // the vector as 4 pairs of fp32 values
  __device__ __forceinline__ static void pairs(const uint4 w, float2* p) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = make_float2(__uint_as_float(u[i] << 16), __uint_as_float(u[i] & 0xFFFF0000u));
  }
  __device__ __forceinline__ static __nv_bfloat162 as2(uint32_t u) {
    return *reinterpret_cast<const __nv_bfloat162*>(&u);
  }
  __device__ __forceinline__ static float at(const void* base, int64_t i) {
    const uint16_t b = reinterpret_cast<const uint16_t*>(base)[i];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
};

template <>
struct Vec16<__half> {
  static constexpr int N = 8;
  static constexpr uint32_t kNegInfWord = 0xFC00FC00u;  // two f16 -inf
  __device__ __forceinline__ static void load(const void* p, float* x) { unpack(*reinterpret_cast<const uint4*>(p), x); }
  __device__ __forceinline__ static void unpack(const uint4 w, float* x) {
    const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ __forceinline__ static void pairs(const uint4 w, float2* p) {
    const __half2* h = reinterpret_cast<const __half2*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __half22float2(h[i]);
  }
  __device__ __forceinline__ static float max8(const uint4* w) {
    const __half2* h = reinterpret_cast<const __half2*>(w);
    __half2 m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2* p = h + 8 * i;
      m[i] = __hmax2(__hmax2(__hmax2(p[0], p[1]), __hmax2(p[2], p[3])),
                     __hmax2(__hmax2(p[4], p[5]), __hmax2(p[6], p[7])));
    }
    const __half2 r = __hmax2(__hmax2(m[0], m[1]), __hmax2(m[2], m[3]));
    return fmaxf(__low2float(r), __high2float(r));
  }
  __device__ __forceinline__ static float at(const void* base, int64_t i) {
    return __half2float(reinterpret_cast<const __half*>(base)[i]);
  }
};

template <>
struct Vec16<float> {
  static constexpr int N = 4;
  static constexpr uint32_t kNegInfWord = 0xFF800000u;
  __device__ __forceinline__ static void load(const void* p, float* x) { unpack(*reinterpret_cast<const uint4*>(p), x); }
  __device__ __forceinline__ static void unpack(const uint4 w, float* x) {
    x[0] = __uint_as_float(w.x);
    x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z);
    x[3] = __uint_as_float(w.w);
  }
  __device__ __forceinline__ static void pairs(const uint4 w, float2* p) {
    p[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
    p[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
  }
  __device__ __forceinline__ static float max8(const uint4* w) {
    float m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 a = w[2 * i], b = w[2 * i + 1];
      m[i] = fmaxf(fmaxf(fmaxf(__uint_as_float(a.x), __uint_as_float(a.y)), fmaxf(__uint_as_float(a.z), __uint_as_float(a.w))),
                   fmaxf(fmaxf(__uint_as_float(b.x), __uint_as_float(b.y)), fmaxf(__uint_as_float(b.z), __uint_as_float(b.w))));
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
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
  int P;               // (m, s) slots per row in the workspace
  int cpr;             // TMA path: chunks per row (a row fills cpr * kTConsumerWarps slots); 0: register path
  bool vec_ok;         // rows and the row length are 16-byte aligned
  const int32_t* sel;
  const int32_t* row_k;
  int k_max;
  Partials parts;
  uint32_t* dev_status;
  uint64_t wait_ns;  // limit of a bounded wait on another role of the CTA
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
  // The chunk just returned by next() was the last of its row piece.
  __device__ bool piece_ended() const { return left == 0 || lb == 0; }
};

// Register path: the (m, s) slot of a row piece, row * P + (range - first range of the row).
__device__ __forceinline__ int64_t piece_slot(const ReduceArgs& a, int row, int range) {
  const int first = static_cast<int>((static_cast<int64_t>(row) * a.nblk) / a.per);
  return static_cast<int64_t>(row) * a.P + (range - first);
}

// ---------------------------------------------------------------------------
// per-row selection
// ---------------------------------------------------------------------------
// select_row() finishes one row from the stream kernel's results: lse from the
// row's (m, s) slots, the selected token's logprob, and the exact top-k.  It is
// run by a group of NT threads (whole warps, ranks tid = 0..NT-1) synchronised
// on named barrier kSelBar: one CTA per row of logits_select_kernel, launched
// after the stream kernel.  (Selecting a row inside the stream kernel, in the
// CTA that completes it, was measured slower: each dependent load of a select
// waits behind the stream's own traffic, and the CTA streams nothing meanwhile.)
// The block maxima, (m, s) slots and selected logit come from the stream
// kernel; they are read through L2 (ld.global.cg).
constexpr int kSelBar = 1;      // named barrier of the selecting group
constexpr int kSThreads = 256;  // logits_select_kernel
constexpr int kSCandCap = 512;  // candidate keys held in shared memory
constexpr int kSKeptCap = 512;  // kept blocks listed per row
constexpr int kSGather = 8;     // candidate vectors per thread in flight

template <int NT>
struct SelectSmem {
  static constexpr int kWarps = NT / 32;
  uint64_t cand[kSCandCap];
  uint32_t hist[256];
  uint32_t misc[4];  // [0] candidates, [1..2] select broadcast, [3] kept blocks
  float wq[kWarps];
  int kept[kSKeptCap];  // the row's kept blocks, in no particular order
  float lse;
};

// Lower bound on the k-th largest logit of a row from its block maxima.
// (m1, m2) are the two largest block maxima of a thread's share of the blocks
// (two distinct blocks); in every warp the q-th largest of the 64 such values
// (q = ceil(k / warps) <= 32) is a value that q distinct blocks of the warp
// reach, so the minimum t over the warps is reached by q * warps >= k distinct
// blocks, each holding a logit >= t: the k-th largest logit is >= t, every
// top-k logit is >= t and lies in a block whose maximum is >= t.  (Two values
// per thread keep t tight when a group of four warps asks for 128.)
template <int NT>
__device__ __forceinline__ float topk_lower_bound(float m1, float m2, int k, float* wq, int tid) {
  constexpr int W = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  const int q = (k + W - 1) / W;
  // the q-th largest of the warp's values: q rounds of (warp max, one holder pops its best)
  uint32_t k1 = f32_ord(m1), k2 = f32_ord(m2);  // > 0 for every value that is not NaN; k1 >= k2
  uint32_t m = 0;
  for (int r = 0; r < q; ++r) {
    m = __reduce_max_sync(0xffffffffu, k1);
    const unsigned holders = __ballot_sync(0xffffffffu, k1 == m);
    if (lane == __ffs(holders) - 1) {
      k1 = k2;
      k2 = 0;  // 0: nothing left in this lane
    }
  }
  if (lane == 0) wq[warp] = ord_f32(m);
  named_bar_sync(kSelBar, NT);
  float t = wq[0];
#pragma unroll
  for (int w = 1; w < W; ++w) t = fminf(t, wq[w]);
  return t;
}

// KB block maxima per thread per round: rows of at most KB * NT blocks take one round,
// their maxima held in registers.
template <typename T, int NT, int KB>
__device__ void select_row(const ReduceArgs& a, int row, int tid, SelectSmem<NT>& sm, float* lse_out,
                           float* sel_logprob, int32_t* topk_ids, float* topk_logprobs) {
  using VT = Vec16<T>;
  constexpr int EPV = VT::N;
  constexpr int VPB = kBlock / EPV;
  const int lane = tid & 31, warp = tid >> 5;
  const int64_t b0 = static_cast<int64_t>(row) * a.nblk;
  // Every independent load first, so that their latencies overlap: the row's
  // block maxima (kept in registers when one round covers the row), its K,
  // the selected token and its logit, and (warp 0) the (m, s) slots.
  const int nb = a.nblk;
  const float* bm = a.parts.bmax + b0;
  const bool one_round = nb <= KB * NT;
  float bv[KB];
  if (one_round) {
#pragma unroll
    for (int i = 0; i < KB; ++i) {
      const int b = tid + i * NT;
      bv[i] = b < nb ? __ldcg(bm + b) : -INFINITY;
    }
  }
  const int k_row = a.row_k ? a.row_k[row] : a.k_max;
  int sel_t = -1;
  float sel_x = 0.0f;
  if (tid == 0 && a.sel) {
    sel_t = a.sel[row];
    sel_x = __ldcg(a.parts.sel_logit + row);  // meaningful only when sel_t is in range
  }
  // (m, s) slots: warp 0 loads them now and folds them into the lse later,
  // off the path to the first barrier (rows of <= 128 slots: one round)
  const int nslots = a.cpr > 0 ? a.cpr * kTConsumerWarps
                               : static_cast<int>((b0 + a.nblk - 1) / a.per - b0 / a.per + 1);
  const float2* ms = a.parts.part_ms + static_cast<int64_t>(row) * a.P;
  float2 msv[4];
  if (warp == 0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = u * 32 + lane;
      msv[u] = j < nslots ? __ldcg(ms + j) : make_float2(-INFINITY, 0.0f);
    }
  }
  // lse = M + log(sum_j s_j exp(m_j - M)); warp 0 writes it (and the selected
  // token's logprob) and leaves it in sm.lse
  auto row_lse = [&]() {
    // two passes over the slots (max, then the rescaled sum): short, parallel dependency chains
    float tm = fmaxf(fmaxf(msv[0].x, msv[1].x), fmaxf(msv[2].x, msv[3].x));
    for (int j = 4 * 32 + lane; j < nslots; j += 32) tm = fmaxf(tm, __ldcg(ms + j).x);
    const float M = warp_max(tm);
    float ts = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int u = 0; u < 4; ++u) ts += msv[u].x == -INFINITY ? 0.0f : msv[u].y * expf(msv[u].x - M);
      for (int j = 4 * 32 + lane; j < nslots; j += 32) {
        const float2 p = __ldcg(ms + j);
        ts += p.x == -INFINITY ? 0.0f : p.y * expf(p.x - M);
      }
    }
    const float S = warp_sum(ts);
    const float lse = (M == -INFINITY) ? -INFINITY : M + logf(S);
    if (lane == 0) {
      sm.lse = lse;
      lse_out[row] = lse;
      if (a.sel) {
        float v = __int_as_float(0x7fc00000);  // NaN: no selected token / out of range
        if (sel_t >= 0 && sel_t < a.V)
          v = sel_x - lse;
        else if (sel_t != -1)
          set_status(a.dev_status, LMH_DS_SEL_OUT_OF_RANGE);
        sel_logprob[row] = v;
      }
    }
  };
  if (tid == 0) {
    sm.misc[0] = 0;
    sm.misc[3] = 0;
  }
  const int k = min(max(k_row, 0), a.k_max);
  if (k == 0) {
    if (warp == 0) row_lse();
    if (a.k_max == 0) return;
    int32_t* out_ids = topk_ids + static_cast<int64_t>(row) * a.k_max;
    float* out_lp = topk_logprobs + static_cast<int64_t>(row) * a.k_max;
    for (int r = tid; r < a.k_max; r += NT) {
      out_ids[r] = -1;
      out_lp[r] = -INFINITY;
    }
    return;
  }

  // ---- t <= the k-th largest logit ----
  // the thread's two largest block maxima (never NaN: fmaxf / fminf drop NaN)
  float m1 = -INFINITY, m2 = -INFINITY;
  auto top2 = [&](float v) {
    m2 = fmaxf(m2, fminf(m1, v));
    m1 = fmaxf(m1, v);
  };
  if (one_round) {
#pragma unroll
    for (int i = 0; i < KB; ++i) top2(bv[i]);
  } else {
    for (int base = 0; base < nb; base += KB * NT) {
      float v[KB];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int b = base + tid + i * NT;
        v[i] = b < nb ? __ldcg(bm + b) : -INFINITY;
      }
#pragma unroll
      for (int i = 0; i < KB; ++i) top2(v[i]);
    }
  }
  const float t = topk_lower_bound<NT>(m1, m2, k, sm.wq, tid);  // (its barrier also publishes misc[0] and misc[3])
  int32_t* out_ids = topk_ids + static_cast<int64_t>(row) * a.k_max;
  float* out_lp = topk_logprobs + static_cast<int64_t>(row) * a.k_max;

  // ---- kept blocks (maximum >= t), one list for the row ----
  const T* rowp = reinterpret_cast<const T*>(a.logits) + static_cast<int64_t>(row) * a.row_stride;
  // a warp places its `mine` blocks (per lane) with one shared atomic; returns the lane's first slot
  auto place = [&](int mine) -> int {
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t wbase = 0;
    if (lane == 31 && total > 0) wbase = atomicAdd(&sm.misc[3], static_cast<uint32_t>(total));
    wbase = __shfl_sync(0xffffffffu, wbase, 31);
    return static_cast<int>(wbase) + incl - mine;
  };
  if (one_round) {
    uint32_t kmask = 0;  // this thread's kept blocks as a bit mask
#pragma unroll
    for (int i = 0; i < KB; ++i) kmask |= ((tid + i * NT < nb && bv[i] >= t) ? 1u : 0u) << i;
    int pos = place(__popc(kmask));
    while (kmask) {
      const int i = __ffs(kmask) - 1;
      kmask &= kmask - 1;
      if (pos < kSKeptCap) sm.kept[pos] = tid + i * NT;
      ++pos;
    }
  } else {
    for (int base = 0; base < nb; base += KB * NT) {
      float v[KB];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const int b = base + tid + i * NT;
        v[i] = b < nb ? __ldcg(bm + b) : -INFINITY;
      }
      uint32_t kmask = 0;
#pragma unroll
      for (int i = 0; i < KB; ++i) kmask |= ((base + tid + i * NT < nb && v[i] >= t) ? 1u : 0u) << i;
      int pos = place(__popc(kmask));
      while (kmask) {
        const int i = __ffs(kmask) - 1;
        kmask &= kmask - 1;
        if (pos < kSKeptCap) sm.kept[pos] = base + tid + i * NT;
        ++pos;
      }
    }
  }
  named_bar_sync(kSelBar, NT);
  const int nkept = static_cast<int>(sm.misc[3]);  // uniform
  auto add_cand = [&](float x, int e) {
    if (x >= t) {
      const uint32_t pos = atomicAdd(&sm.misc[0], 1u);
      if (pos < kSCandCap) sm.cand[pos] = make_key(x, e);
    }
  };
  if (nkept > kSKeptCap) {
    // more kept blocks than the list holds: the exact path below
  } else if (a.vec_ok) {
    // the kept blocks' 16-byte vectors spread evenly over the group, kSGather per thread in
    // flight (one memory round trip for up to NT * kSGather vectors); none straddles the row end.
    // A warp's candidates are placed with one shared atomic: per-lane bit masks and a prefix sum.
    static_assert(kSGather * EPV <= 64, "candidate bit mask");
    const int n_vec = nkept * VPB;
    for (int base = 0; base < n_vec; base += kSGather * NT) {
      uint4 w[kSGather];
      int e0[kSGather];
#pragma unroll
      for (int u = 0; u < kSGather; ++u) {
        const int j = base + u * NT + tid;
        e0[u] = -1;
        if (j < n_vec) {
          const int e = sm.kept[j / VPB] * kBlock + (j % VPB) * EPV;
          if (e < a.V) {
            e0[u] = e;
            w[u] = *reinterpret_cast<const uint4*>(rowp + e);
          }
        }
      }
      uint64_t cmask = 0;  // bit u * EPV + e: element e of vector u reaches t
#pragma unroll
      for (int u = 0; u < kSGather; ++u) {
        float x[EPV];
        VT::unpack(w[u], x);
#pragma unroll
        for (int e = 0; e < EPV; ++e) cmask |= ((e0[u] >= 0 && x[e] >= t) ? 1ull : 0ull) << (u * EPV + e);
      }
      const int mine = __popcll(cmask);
      int incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      uint32_t wbase = 0;
      if (lane == 31 && total > 0) wbase = atomicAdd(&sm.misc[0], static_cast<uint32_t>(total));
      wbase = __shfl_sync(0xffffffffu, wbase, 31);
      uint32_t pos = wbase + static_cast<uint32_t>(incl - mine);
#pragma unroll
      for (int u = 0; u < kSGather; ++u) {
        uint32_t mu = static_cast<uint32_t>(cmask >> (u * EPV)) & ((1u << EPV) - 1u);
        if (!mu) continue;
        float x[EPV];
        VT::unpack(w[u], x);
        while (mu) {
          const int e = __ffs(mu) - 1;
          mu &= mu - 1;
          float v = x[0];  // x[e] without dynamic register indexing
#pragma unroll
          for (int ee = 1; ee < EPV; ++ee) v = (e == ee) ? x[ee] : v;
          if (pos < kSCandCap) sm.cand[pos] = make_key(v, e0[u] + e);
          ++pos;
        }
      }
    }
  } else {
    const int n_el = nkept * kBlock;
    for (int j = tid; j < n_el; j += NT) {
      const int e = sm.kept[j / kBlock] * kBlock + (j % kBlock);
      if (e < a.V) add_cand(VT::at(rowp, e), e);
    }
  }
  if (warp == 0) row_lse();
  named_bar_sync(kSelBar, NT);
  int cnt = static_cast<int>(sm.misc[0]);
  const float lse = sm.lse;
  if (cnt > kSCandCap || nkept > kSKeptCap) {
    // too many entries reach t (ties, rows of -inf): the exact k-th key over
    // them, then the k keys at or above it
    auto in_set = [&](int i, uint64_t* key) -> bool {
      if (i >= a.V || !(__ldcg(bm + i / kBlock) >= t)) return false;
      const float x = VT::at(rowp, i);
      if (!(x >= t)) return false;
      *key = make_key(x, i);
      return true;
    };
    auto sync = [] { named_bar_sync(kSelBar, NT); };
    int above;
    const int n_items = nb * kBlock;
    const uint64_t T64 = group_radix_select(in_set, n_items, k, 64, sm.hist, sm.misc + 1, &above, tid, NT, sync);
    sync();
    if (tid == 0) sm.misc[0] = 0;
    sync();
    for (int i = tid; i < n_items; i += NT) {
      uint64_t key = 0;
      if (in_set(i, &key) && key >= T64) {
        const uint32_t pos = atomicAdd(&sm.misc[0], 1u);  // exactly k of them
        if (pos < kSCandCap) sm.cand[pos] = key;
      }
    }
    sync();
    cnt = min(k, static_cast<int>(sm.misc[0]));
  }
  // ---- exact order (keys are unique) ----
  if (cnt <= 64) {
    // one warp: a bitonic sort of the <= 64 keys, two per lane (key i = lane + 32 h), descending
    if (warp == 0) {
      uint64_t v0 = lane < cnt ? sm.cand[lane] : 0ull, v1 = lane + 32 < cnt ? sm.cand[lane + 32] : 0ull;
#pragma unroll
      for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          if (stride == 32) {  // partners in one lane (size 64: the whole sequence descends)
            const uint64_t hi = v0 > v1 ? v0 : v1, lo = v0 > v1 ? v1 : v0;
            v0 = hi;
            v1 = lo;
          } else {
            const bool lower = (lane & stride) == 0;
            const uint64_t y0 = __shfl_xor_sync(0xffffffffu, v0, stride);
            const uint64_t y1 = __shfl_xor_sync(0xffffffffu, v1, stride);
            const bool d0 = (lane & size) == 0, d1 = ((lane + 32) & size) == 0;  // descending runs
            v0 = (d0 == lower) ? (v0 > y0 ? v0 : y0) : (v0 < y0 ? v0 : y0);
            v1 = (d1 == lower) ? (v1 > y1 ? v1 : y1) : (v1 < y1 ? v1 : y1);
          }
        }
      }
      if (lane < cnt && lane < k) {
        out_ids[lane] = key_id(v0);
        out_lp[lane] = key_value(v0) - lse;
      }
      if (lane + 32 < cnt && lane + 32 < k) {
        out_ids[lane + 32] = key_id(v1);
        out_lp[lane + 32] = key_value(v1) - lse;
      }
    }
  } else {
    // G threads per candidate, each counting the larger keys among a share of the candidates
    int G = 1;  // a power of two <= 32 with G * cnt <= NT, at least 1
    while (G < 32 && 2 * G * cnt <= NT) G *= 2;
    const int groups = NT / G;
    for (int base = 0; base < cnt; base += groups) {
    const int i = base + tid / G, sub = tid % G;
    const uint64_t key = i < cnt ? sm.cand[i] : 0ull;
    int rank = 0;
    if (i < cnt)
      for (int j = sub; j < cnt; j += G) rank += sm.cand[j] > key;
    for (int o = G / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (i < cnt && sub == 0 && rank < k) {
      out_ids[rank] = key_id(key);
      out_lp[rank] = key_value(key) - lse;
    }
    }
  }
  for (int r = min(cnt, k) + tid; r < a.k_max; r += NT) {  // ranks without a candidate, and ranks >= k
    out_ids[r] = -1;
    out_lp[r] = -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// stream kernel, TMA path
// ---------------------------------------------------------------------------
struct StreamDesc {  // one per stage, written by the producer before the copy is issued
  int row;           // < 0: no more chunks
  int lb;            // first 64-block of the chunk within the row
  int nbk;           // blocks in the chunk
  int ne;            // real logits in the chunk (the copied ones)
  int64_t slot;      // first (m, s) slot of the chunk: one per consumer warp
  int sel_rel;       // selected token relative to the chunk's first logit
};
static_assert(sizeof(StreamDesc) <= kTDescBytes, "descriptor slot");

constexpr int kTSmem = kTSmemRing;

template <typename T>
__global__ void __launch_bounds__(kTThreads, kTCtasPerSm) logits_stream_tma_kernel(const ReduceArgs a) {
  using VT = Vec16<T>;
  constexpr int ES = static_cast<int>(sizeof(T));
  constexpr int EPV = VT::N;         // elements per 16-byte vector
  constexpr int EPT = 128 / ES;      // elements per consumer thread
  constexpr int TPB = kBlock / EPT;  // consumer threads per 64-block (1, or 2 for f32)
  constexpr int CH = kTConsumers / TPB;  // blocks per chunk
  constexpr int S = kTStages;

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stages = smem;
  StreamDesc* desc = reinterpret_cast<StreamDesc*>(smem + S * kTChunkBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * kTChunkBytes + S * kTDescBytes);
  uint64_t* empty = full + S;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTConsumerWarps);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_launch_dependents();  // the select kernel may be scheduled; it waits for this grid's results

  if (warp == kTConsumerWarps) {
    // ------------------------------ producer ------------------------------
    // Chunks (CH blocks of one row; chunk c is row c / cpr, part c % cpr) are
    // handed out dynamically, so CTAs that stream faster take more of them:
    // the first S of a CTA are fixed (blockIdx.x + j * gridDim.x), the rest
    // come from the ticket counter (draws base + 0, 1, ...), drawn one chunk
    // ahead.  Without a valid base (TicketState) every chunk is fixed.
    if (lane != 0) return;
    const int64_t total = static_cast<int64_t>(a.rows) * a.cpr;
    const int64_t first_dynamic = static_cast<int64_t>(S) * gridDim.x;
    const uint64_t policy = l2_evict_first_policy();  // logits are read once; the block maxima stay in L2
    int sel_row = -1, sel_id = -1;
    // Stage s <- chunk c (false: c is past the end, and stage s gets the end marker).
    auto issue = [&](int s, int64_t c) {
      StreamDesc& d = desc[s];
      if (c >= total) {
        d.row = -1;
        mbar_arrive(&full[s]);  // end marker: completes with no bytes
        return false;
      }
      const int row = static_cast<int>(c / a.cpr);
      const int ci = static_cast<int>(c - static_cast<int64_t>(row) * a.cpr);
      const int lb = ci * CH;
      const int nbk = min(CH, a.nblk - lb);
      if (row != sel_row) {
        sel_row = row;
        sel_id = a.sel ? a.sel[row] : -1;
      }
      const int ne = min(nbk * kBlock, a.V - lb * kBlock);
      d.row = row;
      d.lb = lb;
      d.nbk = nbk;
      d.ne = ne;
      d.slot = static_cast<int64_t>(row) * a.P + static_cast<int64_t>(ci) * kTConsumerWarps;
      d.sel_rel = sel_id - lb * kBlock;
      const char* src = a.logits + (static_cast<int64_t>(row) * a.row_stride + static_cast<int64_t>(lb) * kBlock) * ES;
      mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(ne * ES));
      bulk_load_hint(stages + static_cast<size_t>(s) * kTChunkBytes, src, static_cast<uint32_t>(ne * ES), &full[s],
                     policy);
      return true;
    };
    // A CTA's first S chunks are fixed: they go out before the grid-dependency wait, so
    // they stream while the kernel before this one (the previous call's select kernel)
    // still runs.  They read only the call's inputs, which were complete before that
    // kernel left its own wait; the workspace (the ticket, the partials) is touched
    // only after this kernel's wait, and the consumers wait too before writing it.
    uint32_t issued = 0;
    bool ended = false;
    for (; issued < static_cast<uint32_t>(S) && !ended; ++issued)
      ended = !issue(static_cast<int>(issued), blockIdx.x + static_cast<int64_t>(issued) * gridDim.x);
    pdl_wait();
    // Read through L2 (another kernel wrote them; an L1 line of an earlier call could be stale).
    TicketState* tk = a.parts.ticket;
    const unsigned long long base = __ldcg(&tk->base);
    const bool dynamic = __ldcg(&tk->check) == ~base;  // the same in every CTA: nothing writes these now
    auto draw = [&](uint32_t n) -> int64_t {  // the chunk of this CTA's n-th load (n >= S)
      return !dynamic ? blockIdx.x + static_cast<int64_t>(n) * gridDim.x
                      : first_dynamic + static_cast<int64_t>(atomicAdd(&tk->ticket, 1ull) - base);
    };
    int64_t next = ended ? total : draw(issued);  // drawn one chunk ahead
    for (; !ended; ++issued) {
      const int s = static_cast<int>(issued % S);
      if (!wait_or_abort(&empty[s], ((issued / S) & 1u) ^ 1u, abort_flag, a.dev_status, a.wait_ns)) break;
      const int64_t c = next;
      if (c < total) next = draw(issued + 1);
      ended = !issue(s, c);
    }
    // Copies still in flight (only after an abort) land before the CTA exits;
    // these waits keep the full limit whatever a.wait_ns is.
    const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
    for (uint32_t i = first; i < issued; ++i) mbar_wait(&full[i % S], (i / S) & 1u);
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int c = tid;  // consumer thread 0..127: bytes [128c, 128c + 128) of a chunk
  const int rot = c & 7;  // vector order rotated by lane: conflict-free 16-byte shared loads
  // The block maxima are read back by the select kernel right after this one: they stay in
  // L2 (evict-last) while the logits, read once, go first (evict-first).
  const uint64_t keep_policy = l2_evict_last_policy();
  const int bi = c / TPB;
  const float L = kLog2e;
  pdl_wait();  // the stages may fill before the kernel before this one ends; the workspace may not be written
  for (uint32_t i = 0;; ++i) {
    const int s = static_cast<int>(i % S);
    const bool ok = wait_or_abort(&full[s], (i / S) & 1u, abort_flag, a.dev_status, a.wait_ns);
    if (!__all_sync(0xffffffffu, ok)) break;
    const StreamDesc d = desc[s];
    if (d.row < 0) break;
    const unsigned char* stg = stages + static_cast<size_t>(s) * kTChunkBytes;
    uint4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = *reinterpret_cast<const uint4*>(stg + c * 128 + ((j + rot) & 7) * 16);
    const bool sel_hit = static_cast<unsigned>(d.sel_rel - c * EPT) < static_cast<unsigned>(EPT) && d.sel_rel < d.ne;
    float selv = 0.0f;
    if (sel_hit) selv = VT::at(stg, d.sel_rel);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the stage is in registers: release it
    if (sel_hit) a.parts.sel_logit[d.row] = selv;

    const int ne_t = d.ne - c * EPT;  // real logits among this thread's
    if (ne_t < EPT) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (((j + rot) & 7) * EPV >= ne_t)
          w[j] = make_uint4(VT::kNegInfWord, VT::kNegInfWord, VT::kNegInfWord, VT::kNegInfWord);
    }
    const float vm = VT::max8(w);  // this thread's maximum
    float bmx = vm;
    if (TPB == 2) bmx = fmaxf(bmx, __shfl_xor_sync(0xffffffffu, bmx, 1));
    if ((c % TPB) == 0 && bi < d.nbk)
      st_keep(a.parts.bmax + static_cast<int64_t>(d.row) * a.nblk + d.lb + bi, bmx, keep_policy);
    float ts = 0.0f;  // sum of exp(x - vm) over this thread's logits
    if (vm > -INFINITY) {
      // exp(x - m) = 2^(x*log2e - m*log2e): one packed FFMA2 and one packed
      // FADD2 per pair of logits around the two ex2
      const float2 L2 = make_float2(L, L), nmL2 = make_float2(-vm * L, -vm * L);
      float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                       make_float2(0.0f, 0.0f)};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float2 p[EPV / 2];
        VT::pairs(w[j], p);
#pragma unroll
        for (int q = 0; q < EPV / 2; ++q) {
          const float2 y = __ffma2_rn(p[q], L2, nmL2);
          acc[q & 3] = __fadd2_rn(acc[q & 3], make_float2(ex2_approx(y.x), ex2_approx(y.y)));
        }
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 a = __fadd2_rn(a01, a23);
      ts = a.x + a.y;
    }
    // the warp's (m, s) over this chunk
    const float M = warp_max(vm);
    const float sc = warp_sum(vm == -INFINITY ? 0.0f : ts * ex2_approx((vm - M) * L));
    if (lane == 0) a.parts.part_ms[d.slot + warp] = make_float2(M, M == -INFINITY ? 0.0f : sc);
  }
}

// ---------------------------------------------------------------------------
// stream kernel, register path (any element-aligned layout)
// ---------------------------------------------------------------------------

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
__global__ void __launch_bounds__(kRThreads, kRCtasPerSm) logits_stream_regs_kernel(const ReduceArgs a) {
  using VT = Vec16<T>;
  constexpr int EPV = VT::N;                            // elements per 16-byte vector
  constexpr int VPB = kBlock / EPV;                     // vectors per 64-block
  constexpr int CH = kRVecPerThread * kRThreads / VPB;  // blocks per chunk

  __shared__ float red[32];
  pdl_launch_dependents();  // the select kernel may be scheduled now; it waits for this grid's results

  ChunkIter<CH> it;
  it.init(a);
  Chunk cur = it.next(a);
  bool cur_end = it.piece_ended();
  ChunkRegs<T> buf0, buf1;  // two register buffers with fixed roles per half of the unrolled loop
  if (cur.valid) buf0.load(a, cur);

  const float L = kLog2e;
  float tm = -INFINITY, ts = 0.0f;  // this thread's running max / sum over the current piece
  int sel_row = -1, sel_id = -1;
  auto step = [&](ChunkRegs<T>& cb, ChunkRegs<T>& nb) {
    const Chunk nxt = it.next(a);
    const bool nxt_end = it.piece_ended();
    if (nxt.valid) nb.load(a, nxt);  // in flight while this chunk is worked on
    if (cur.row != sel_row) {
      sel_row = cur.row;
      sel_id = a.sel ? a.sel[cur.row] : -1;
    }
    const int ne = cb.ne;
    const int rel0 = sel_id - cur.lb * kBlock;  // selected token relative to this chunk
    const bool sel_here = rel0 >= 0 && rel0 < ne;

    // ---- block maxima + online (m, s) ----
#pragma unroll
    for (int j = 0; j < kRVecPerThread; ++j) {
      const int v = threadIdx.x + j * kRThreads;
      float x[EPV];
      VT::unpack(cb.w[j], x);
      float vm = x[0];
#pragma unroll
      for (int e = 1; e < EPV; ++e) vm = fmaxf(vm, x[e]);
      if (vm > tm) {
        ts *= ex2_approx((tm - vm) * L);  // tm = -inf: ts is 0 and stays 0
        tm = vm;
      }
      if (tm != -INFINITY) {
        const float mL = tm * L;
#pragma unroll
        for (int e = 0; e < EPV; ++e) ts += ex2_approx(fmaf(x[e], L, -mL));
      }
      if (sel_here) {
        const unsigned r = static_cast<unsigned>(rel0 - v * EPV);
        if (r < static_cast<unsigned>(EPV)) {
          float sv = 0.0f;
#pragma unroll
          for (int e = 0; e < EPV; ++e) sv = (static_cast<unsigned>(e) == r) ? x[e] : sv;
          a.parts.sel_logit[cur.row] = sv;
        }
      }
#pragma unroll
      for (int o = VPB / 2; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
      if (v * EPV < cur.nbk * kBlock && (threadIdx.x % VPB) == 0)
        a.parts.bmax[static_cast<int64_t>(cur.row) * a.nblk + cur.lb + v / VPB] = vm;
    }

    if (cur_end) {
      const float M = block_max(tm, red);
      const float S = block_sum((tm == -INFINITY) ? 0.0f : ts * ex2_approx((tm - M) * L), red);
      if (threadIdx.x == 0) a.parts.part_ms[piece_slot(a, cur.row, cur.range)] = make_float2(M, M == -INFINITY ? 0.0f : S);
      tm = -INFINITY;
      ts = 0.0f;
    }
    cur = nxt;
    cur_end = nxt_end;
  };
  while (cur.valid) {
    step(buf0, buf1);
    if (!cur.valid) break;
    step(buf1, buf0);
  }
}

// The per-row select: one CTA per row, after the stream kernel.
template <typename T>
__global__ void __launch_bounds__(kSThreads) logits_select_kernel(const ReduceArgs a, float* lse_out,
                                                                  float* sel_logprob, int32_t* topk_ids,
                                                                  float* topk_logprobs) {
  __shared__ SelectSmem<kSThreads> sm;
  pdl_wait();  // the block maxima and (m, s) come from the stream kernel just before
  pdl_launch_dependents();  // a following kernel may be scheduled; it waits for this grid before using its results
  if (blockIdx.x == 0 && threadIdx.x == 0) {  // the stream kernel is done with the ticket: the next call's base
    TicketState* tk = a.parts.ticket;
    const unsigned long long t = __ldcg(&tk->ticket);  // through L2: the stream kernel's atomics wrote it
    tk->base = t;
    tk->check = ~t;
  }
  select_row<T, kSThreads, 16>(a, blockIdx.x, threadIdx.x, sm, lse_out, sel_logprob, topk_ids, topk_logprobs);
}

// ---------------------------------------------------------------------------
// full-vocabulary output (k_max = LMH_K_FULL)
// ---------------------------------------------------------------------------
// out[r][v] = fp32(x[r][v]) - lse[r] for every id: one coalesced pass, 8
// elements per thread, reads x, writes f32.  `x` may be `out` itself (the
// head path materializes its fp32 logits there first).
constexpr int kFThreads = 256;
constexpr int kFPerThread = 8;

template <typename T>
__global__ void __launch_bounds__(kFThreads) full_logprobs_kernel(const T* x, int64_t row_stride, int V,
                                                                   const float* __restrict__ lse, float* out) {
  pdl_wait();  // lse (and in place, the logits) come from the kernels launched just before
  const int row = blockIdx.x;  // rows on x (no 65535 limit), column chunks on y
  const float l = lse[row];
  const T* src = x + static_cast<int64_t>(row) * row_stride;
  float* dst = out + static_cast<int64_t>(row) * V;
  const int base = blockIdx.y * (kFThreads * kFPerThread) + threadIdx.x;
  float v[kFPerThread];
#pragma unroll
  for (int u = 0; u < kFPerThread; ++u) {
    const int c = base + u * kFThreads;
    v[u] = c < V ? Vec16<T>::at(src, c) : 0.0f;
  }
#pragma unroll
  for (int u = 0; u < kFPerThread; ++u) {
    const int c = base + u * kFThreads;
    if (c < V) dst[c] = v[u] - l;
  }
}

cudaError_t launch_full_logprobs(const void* x, lmh_dtype dtype, int64_t row_stride, int rows, int V, const float* lse,
                                 float* out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const dim3 grid(rows, (V + kFThreads * kFPerThread - 1) / (kFThreads * kFPerThread));
  cudaError_t e;
  trace_begin(kTraceFull, stream);
  switch (dtype) {
    case LMH_BF16:
      e = launch_kernel(full_logprobs_kernel<__nv_bfloat16>, grid, dim3(kFThreads), 0, stream, true,
                        static_cast<const __nv_bfloat16*>(x), row_stride, V, lse, out);
      break;
    case LMH_F16:
      e = launch_kernel(full_logprobs_kernel<__half>, grid, dim3(kFThreads), 0, stream, true,
                        static_cast<const __half*>(x), row_stride, V, lse, out);
      break;
    default:
      e = launch_kernel(full_logprobs_kernel<float>, grid, dim3(kFThreads), 0, stream, true,
                        static_cast<const float*>(x), row_stride, V, lse, out);
      break;
  }
  trace_end(kTraceFull, stream);
  return e;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

VocabSplit logits_reduce_split(int rows, int V, int k_max, int num_sms) {
  VocabSplit vs;
  const int nblk = (V + kBlock - 1) / kBlock;
  const int64_t nb_total = static_cast<int64_t>(rows) * nblk;
  const int sms = num_sms > 0 ? num_sms : 1;
  const int64_t G = static_cast<int64_t>(sms) * kRCtasPerSm;  // ranges aimed at: two per SM
  int64_t per = (nb_total + G - 1) / G;
  // a range of more than 2k blocks lets the block-max threshold prune (<= k blocks keep everything)
  const int64_t min_per = 2 * k_max > kRMinPer ? 2 * k_max : kRMinPer;
  if (per < min_per) per = min_per;
  if (per > kRMaxPer) per = kRMaxPer;
  vs.per = static_cast<int>(per);
  vs.n_ranges = static_cast<int>((nb_total + per - 1) / per);
  vs.grid = static_cast<int>(vs.n_ranges < G ? vs.n_ranges : G);
  vs.ctas = sms * kTCtasPerSm;
  vs.splits = static_cast<int>((nblk + per - 1) / per) + 1;  // row pieces per row, at most
  vs.nblk = nblk;
  // TMA path: one slot per consumer warp and chunk; the smallest chunk (f32) has kTChunkBytes / 256 blocks
  const int cpr_max = (nblk + kTChunkBytes / 256 - 1) / (kTChunkBytes / 256);
  vs.slots = cpr_max * kTConsumerWarps > vs.splits ? cpr_max * kTConsumerWarps : vs.splits;
  return vs;
}

template <typename T>
static cudaError_t setup_one() {
  cudaError_t e =
      cudaFuncSetAttribute(logits_stream_tma_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem);
  // Both kernels ask for the largest shared-memory carveout, so that the SMs
  // keep one L1 / shared split from one kernel to the next.
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(logits_stream_tma_kernel<T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(logits_select_kernel<T>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t logits_reduce_setup() {
  cudaError_t e = setup_one<__nv_bfloat16>();
  if (e == cudaSuccess) e = setup_one<__half>();
  if (e == cudaSuccess) e = setup_one<float>();
  return e;
}

size_t stream_partials_bytes(int rows, const VocabSplit& vs) {
  auto al = [](size_t n) { return (n + 255) & ~static_cast<size_t>(255); };
  return al(static_cast<size_t>(rows) * vs.slots * 8) + al(static_cast<size_t>(rows) * 4) +
         al(static_cast<size_t>(rows) * vs.nblk * 4) + al(sizeof(TicketState));
}

Partials carve_stream_partials(void* base, int rows, const VocabSplit& vs) {
  auto al = [](size_t n) { return (n + 255) & ~static_cast<size_t>(255); };
  char* p = static_cast<char*>(base);
  Partials out;
  out.part_ms = reinterpret_cast<float2*>(p);
  p += al(static_cast<size_t>(rows) * vs.slots * 8);
  out.sel_logit = reinterpret_cast<float*>(p);
  p += al(static_cast<size_t>(rows) * 4);
  out.bmax = reinterpret_cast<float*>(p);
  p += al(static_cast<size_t>(rows) * vs.nblk * 4);
  out.ticket = reinterpret_cast<TicketState*>(p);
  out.part_keys = nullptr;
  out.part_samp = nullptr;
  return out;
}

template <typename T>
static cudaError_t launch_both(ReduceArgs a, const VocabSplit& split, float* lse, float* sel_logprob,
                               int32_t* topk_ids, float* topk_logprobs, cudaStream_t stream) {
  cudaError_t e;
  if (a.vec_ok) {
    constexpr int CH = kTChunkBytes / (kBlock * static_cast<int>(sizeof(T)));  // blocks per chunk
    a.cpr = (a.nblk + CH - 1) / CH;
    const int64_t chunks = static_cast<int64_t>(a.rows) * a.cpr;
    const int grid = static_cast<int>(chunks < split.ctas ? chunks : split.ctas);
    trace_begin(kTraceReduce, stream);
    e = launch_kernel(logits_stream_tma_kernel<T>, dim3(grid), dim3(kTThreads), static_cast<size_t>(kTSmem), stream,
                      true, a);
  } else {
    a.cpr = 0;
    trace_begin(kTraceReduce, stream);
    e = launch_kernel(logits_stream_regs_kernel<T>, dim3(split.grid), dim3(kRThreads), 0, stream, false, a);
  }
  trace_end(kTraceReduce, stream);
  if (e != cudaSuccess) return e;
  trace_begin(kTraceLogitsSelect, stream);
  e = launch_kernel(logits_select_kernel<T>, dim3(a.rows), dim3(kSThreads), 0, stream, true, a, lse, sel_logprob,
                    topk_ids, topk_logprobs);
  trace_end(kTraceLogitsSelect, stream);
  return e;
}

cudaError_t launch_logits_reduce(const void* logits, lmh_dtype dtype, int64_t row_stride, int rows, int V,
                                 VocabSplit split, const int32_t* sel, const int32_t* row_k, int k_max,
                                 Partials parts, float* lse, float* sel_logprob, int32_t* topk_ids,
                                 float* topk_logprobs, uint32_t* dev_status, cudaStream_t stream) {
  // Full-vocabulary output: the reduction with K 0 (lse, selected token), then z - lse for every id.
  const bool full = k_max == LMH_K_FULL;
  if (full) k_max = 0;
  const int64_t es = dtype == LMH_F32 ? 4 : 2;
  ReduceArgs a;
  a.logits = static_cast<const char*>(logits);
  a.row_stride = row_stride;
  a.rows = rows;
  a.V = V;
  a.nblk = split.nblk;
  a.nb_total = static_cast<int64_t>(rows) * split.nblk;
  a.per = split.per;
  a.n_ranges = split.n_ranges;
  a.P = split.slots;
  a.cpr = 0;
  a.vec_ok = (reinterpret_cast<uintptr_t>(logits) % 16) == 0 && ((row_stride * es) % 16) == 0 &&
             ((static_cast<int64_t>(V) * es) % 16) == 0;
  a.sel = sel;
  a.row_k = row_k;
  a.k_max = k_max;
  a.parts = parts;
  a.dev_status = dev_status;
  a.wait_ns = wait_limit_ns();
  cudaError_t e;
  switch (dtype) {
    case LMH_BF16:
      e = launch_both<__nv_bfloat16>(a, split, lse, sel_logprob, topk_ids, topk_logprobs, stream);
      break;
    case LMH_F16:
      e = launch_both<__half>(a, split, lse, sel_logprob, topk_ids, topk_logprobs, stream);
      break;
    default:
      e = launch_both<float>(a, split, lse, sel_logprob, topk_ids, topk_logprobs, stream);
      break;
  }
  if (e == cudaSuccess && full) e = launch_full_logprobs(logits, dtype, row_stride, rows, V, lse, topk_logprobs, stream);
  return e;
}

}  // namespace lmh
