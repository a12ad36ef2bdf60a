// merge_partials.cu -- combine the per-chunk partials of every row (K5).
//
// openinfer issue #719, "Suggested direction": a numerically sound
// multi-stage reduction that returns lse, the selected-token logprob and the
// top-k as an O(k+1) result.  MTPLX PR #532, "Change": logprob = fp32(logit)
// - lse, evaluated only at the survivors and at the scored token; exact ties
// by ascending id.
//
// One CTA per row (merge_partials_kernel), or one warp per row when a row has at
// most 128 slots (merge_partials_slots_kernel) or its slots hold few keys
// (merge_partials_warp_kernel).
#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

constexpr int kMergeThreads = 256;
constexpr int kMergeCap = 1024;  // candidate keys held in shared memory

struct MergeArgs {
  int rows, splits, V, k_max;
  Partials parts;
  const int32_t* sel;
  const int32_t* row_k;
  float* lse;
  float* sel_logprob;
  int32_t* topk_ids;
  float* topk_logprobs;
  uint32_t* dev_status;
  SampleArgs samp;
  RecordOut rec;  // rec.base != null: write each row's vocabulary-parallel record instead of results
};

// The row's record (vocabulary-parallel share) and its keys.
__device__ __forceinline__ VocabRecord* row_record(const MergeArgs& a, int row) {
  return reinterpret_cast<VocabRecord*>(a.rec.base + static_cast<int64_t>(row) * record_bytes(a.k_max));
}
__device__ __forceinline__ unsigned long long* record_keys(VocabRecord* r) {
  return reinterpret_cast<unsigned long long*>(r + 1);
}

// Record mode: the share's (M, S), and the selected logit when the token lies in the share.
__device__ __forceinline__ void write_record_head(const MergeArgs& a, int row, float M, float S) {
  VocabRecord* r = row_record(a, row);
  const int t = a.sel ? a.sel[row] : -1;
  const bool has = t >= a.rec.v_begin && t < a.rec.v_begin + a.rec.v_count;
  r->m = M;
  r->s = M == -INFINITY ? 0.0f : S;
  r->sel_logit = has ? a.parts.sel_logit[row] : 0.0f;
  r->flags = has ? kRecordHasSel : 0u;
}

// Sampling partials (score, id bits, z, -): a beats b when it has a token and a
// higher score, ties to the smaller id (the order in which one stream meets them).
__device__ __forceinline__ bool samp_better(const float4& a, const float4& b) {
  const int ia = __float_as_int(a.y), ib = __float_as_int(b.y);
  if (ia < 0) return false;
  if (ib < 0) return true;
  return a.x > b.x || (a.x == b.x && ia < ib);
}

__device__ __forceinline__ float4 samp_warp_best(float4 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float4 w;
    w.x = __shfl_xor_sync(0xffffffffu, v.x, o);
    w.y = __shfl_xor_sync(0xffffffffu, v.y, o);
    w.z = __shfl_xor_sync(0xffffffffu, v.z, o);
    w.w = 0.0f;
    if (samp_better(w, v)) v = w;
  }
  return v;
}

// The row's sampled token from its slots' partials; writes id and z - lse.
__device__ __forceinline__ void samp_write(const MergeArgs& a, int row, float4 best, float lse) {
  const int id = __float_as_int(best.y);
  a.samp.ids_out[row] = id;
  if (a.samp.lp_out) a.samp.lp_out[row] = id >= 0 ? best.z - lse : __int_as_float(0x7fc00000);
  if (id < 0) set_status(a.dev_status, LMH_DS_NO_ALLOWED_TOKEN);
}

// One CTA per row:
//   lse = M + log(sum_j s_j * exp(m_j - M)) over the row's slots j, with
//         M = max_j m_j (lse = -inf when every logit is -inf);
//   top-k = the k best keys of the union of the slots' sorted top-k lists.
//         Every slot list holds that piece's k best, so the union holds the
//         row's k best.  A lower bound L of the row's k-th key (the minimum
//         over the warps of each warp's q-th largest held list value, q =
//         ceil(k / warps)) limits the gather to keys >= L;
//         they are ordered by rank.
// The best of a row's slot partials, by the whole CTA (kept out of line so
// that its registers do not add to the merge's).
__device__ __noinline__ void cta_sample(const MergeArgs& a, int row, int nslots, float lse) {
  __shared__ float4 s_samp[kMergeThreads / 32];
  const int tid = threadIdx.x;
  const float4* ps = a.parts.part_samp + static_cast<int64_t>(row) * nslots;
  float4 b = make_float4(-INFINITY, __int_as_float(-1), -INFINITY, 0.0f);
  for (int j = tid; j < nslots; j += kMergeThreads) {
    const float4 c = ps[j];
    if (samp_better(c, b)) b = c;
  }
  b = samp_warp_best(b);
  if ((tid & 31) == 0) s_samp[tid >> 5] = b;
  __syncthreads();
  if (tid == 0) {
    float4 r = s_samp[0];
    for (int w = 1; w < kMergeThreads / 32; ++w)
      if (samp_better(s_samp[w], r)) r = s_samp[w];
    samp_write(a, row, r, lse);
  }
}

constexpr int kMergeItemsPerThread = 12;  // a row's keys held in registers per thread (first round)

__global__ void __launch_bounds__(kMergeThreads, 4) merge_partials_kernel(const MergeArgs a) {
  __shared__ uint64_t cand[kMergeCap];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t misc[4];  // [0] candidates, [1..2] select broadcast
  __shared__ float red[32];
  __shared__ uint32_t lbw[kMergeThreads / 32];  // per-warp bounds (read once, after one barrier)
  pdl_wait();  // the partials come from the kernel launched just before
  pdl_launch_dependents();  // a following kernel may be scheduled; it waits for this grid before using its results
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int nslots = a.splits;
  const float2* ms = a.parts.part_ms + static_cast<int64_t>(row) * nslots;
  const unsigned long long* keys = a.parts.part_keys + static_cast<int64_t>(row) * nslots * a.k_max;

  // ---- every independent load first: K, the selected token, the slots' (m, s) and the row's keys ----
  // Slot j's sorted list is keys[j * k_max + r], r < k_max: item i = j * k_max + r is keys[i].
  const int k = a.row_k ? min(max(a.row_k[row], 0), a.k_max) : a.k_max;
  int sel_t = -1;
  float sel_x = 0.0f;
  if (tid == 0 && a.sel) {
    sel_t = a.sel[row];
    sel_x = a.parts.sel_logit[row];  // meaningful only when sel_t is in range
  }
  const float2 p0 = tid < nslots ? ms[tid] : make_float2(-INFINITY, 0.0f);
  const int n_items = nslots * a.k_max;
  uint64_t kv[kMergeItemsPerThread];
#pragma unroll
  for (int u = 0; u < kMergeItemsPerThread; ++u) {
    const int i = tid + u * kMergeThreads;
    kv[u] = i < n_items ? keys[i] : 0ull;
  }
  // (slot, rank) of the held items, walked without divisions
  const int km = max(a.k_max, 1);
  const int step_j = kMergeThreads / km, step_r = kMergeThreads - step_j * km;
  const int j0 = tid / km, r0 = tid - j0 * km;
  auto next = [&](int& j, int& r) {
    j += step_j;
    r += step_r;
    if (r >= km) {
      r -= km;
      ++j;
    }
  };

  // ---- lse = M + log(sum_j s_j exp(m_j - M)) ----
  float mloc = p0.x;
  for (int j = tid + kMergeThreads; j < nslots; j += kMergeThreads) mloc = fmaxf(mloc, ms[j].x);
  const float M = block_max(mloc, red);
  float sloc = 0.0f;
  if (M != -INFINITY) {
    if (p0.x != -INFINITY) sloc = p0.y * expf(p0.x - M);
    for (int j = tid + kMergeThreads; j < nslots; j += kMergeThreads) {
      const float2 p = ms[j];
      if (p.x != -INFINITY) sloc += p.y * expf(p.x - M);
    }
  }
  const float S = block_sum(sloc, red);
  const float lse = (M == -INFINITY) ? -INFINITY : M + logf(S);
  const bool rec_mode = a.rec.base != nullptr;
  if (tid == 0 && rec_mode) {
    write_record_head(a, row, M, S);
    misc[0] = 0;
  } else if (tid == 0) {
    a.lse[row] = lse;
    if (a.sel) {
      float v = __int_as_float(0x7fc00000);  // NaN: no selected token / out of range
      if (sel_t >= 0 && sel_t < a.V)
        v = sel_x - lse;
      else if (sel_t != -1)
        set_status(a.dev_status, LMH_DS_SEL_OUT_OF_RANGE);
      a.sel_logprob[row] = v;
    }
    misc[0] = 0;
  }
  if (a.samp.enabled) cta_sample(a, row, nslots, lse);  // the sampled token: the best slot partial
  if (a.k_max == 0) return;
  int32_t* out_ids = rec_mode ? nullptr : a.topk_ids + static_cast<int64_t>(row) * a.k_max;
  float* out_lp = rec_mode ? nullptr : a.topk_logprobs + static_cast<int64_t>(row) * a.k_max;
  unsigned long long* out_keys = rec_mode ? record_keys(row_record(a, row)) : nullptr;
  // rank r: the key (record mode) or its id and logprob (key 0: no entry)
  auto put = [&](int r, uint64_t key) {
    if (rec_mode) {
      out_keys[r] = key;
    } else {
      out_ids[r] = key ? key_id(key) : -1;
      out_lp[r] = key ? key_value(key) - lse : -INFINITY;
    }
  };
  if (k == 0) {
    for (int r = tid; r < a.k_max; r += kMergeThreads) put(r, 0ull);
    return;
  }

  // ---- lb: a lower bound of the row's k-th key ----
  // The first k entries of a slot's list are logits of the row (the slot's best k; the
  // entries past the row's K are not written).  Every warp takes the q-th largest value
  // among such keys its threads hold (q = ceil(k / warps): q rounds of a warp-wide max,
  // one holder of the maximum dropping out each round); the minimum t over the warps is
  // reached by q * warps >= k logits of the row, so the row's k-th key has a value >= t
  // and every top-k key is >= (t, any id).  A warp holding fewer than q keys gives t = 0:
  // no pruning.
  uint64_t lb = 0;
  {
    constexpr int kWarps = kMergeThreads / 32;
    const int q = (k + kWarps - 1) / kWarps;
    uint32_t uv[kMergeItemsPerThread];  // ordered values of the held keys (0: none)
    int j = j0, r = r0;
#pragma unroll
    for (int u = 0; u < kMergeItemsPerThread; ++u) {
      uv[u] = r < k ? static_cast<uint32_t>(kv[u] >> 32) : 0u;  // kv is 0 past the row's items
      next(j, r);
    }
    const int lane = tid & 31;
    uint32_t t = 0;
    for (int round = 0; round < q; ++round) {
      uint32_t mine = 0;
#pragma unroll
      for (int u = 0; u < kMergeItemsPerThread; ++u) mine = max(mine, uv[u]);
      const uint32_t wmax = __reduce_max_sync(0xffffffffu, mine);
      t = wmax;
      if (wmax == 0u) break;  // fewer than q held keys in this warp
      const unsigned holders = __ballot_sync(0xffffffffu, mine == wmax);
      if (lane == __ffs(holders) - 1) {  // drop one instance of the maximum
        bool done = false;
#pragma unroll
        for (int u = 0; u < kMergeItemsPerThread; ++u) {
          const bool hit = !done && uv[u] == wmax;
          uv[u] = hit ? 0u : uv[u];
          done = done || hit;
        }
      }
    }
    if (lane == 0) lbw[tid >> 5] = t;
    __syncthreads();
    uint32_t tmin = 0xFFFFFFFFu;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tmin = min(tmin, lbw[w]);
    lb = static_cast<uint64_t>(tmin) << 32;
  }

  // ---- candidates: the keys >= lb among the first k of every slot ----
  auto take = [&](int i, uint64_t key) {
    const int r = i % a.k_max;
    if (r < k && key != 0ull && key >= lb) {
      const uint32_t pos = atomicAdd(&misc[0], 1u);
      if (pos < kMergeCap) cand[pos] = key;
    }
  };
  {
    int j = j0, r = r0;
#pragma unroll
    for (int u = 0; u < kMergeItemsPerThread; ++u) {
      const uint64_t key = kv[u];  // 0 beyond n_items
      if (r < k && key != 0ull && key >= lb) {
        const uint32_t pos = atomicAdd(&misc[0], 1u);
        if (pos < kMergeCap) cand[pos] = key;
      }
      next(j, r);
    }
  }
  for (int i = tid + kMergeItemsPerThread * kMergeThreads; i < n_items; i += kMergeThreads) take(i, keys[i]);
  __syncthreads();
  int cnt = static_cast<int>(misc[0]);
  if (cnt > kMergeCap) {
    // many exact ties: select the k-th key exactly, then keep the k keys at or above it
    const int n_set = nslots * k;
    auto in_set = [&](int i, uint64_t* key) -> bool {
      const int j = i / k, r = i - j * k;
      const uint64_t kk = keys[static_cast<int64_t>(j) * a.k_max + r];
      if (kk == 0ull || kk < lb) return false;
      *key = kk;
      return true;
    };
    int above;
    const uint64_t T64 = cta_radix_select(in_set, n_set, k, 64, hist, misc + 1, &above);
    __syncthreads();
    if (tid == 0) misc[0] = 0;
    __syncthreads();
    for (int i = tid; i < n_set; i += kMergeThreads) {
      uint64_t key = 0;
      if (in_set(i, &key) && key >= T64) {
        const uint32_t pos = atomicAdd(&misc[0], 1u);  // exactly k of them
        if (pos < kMergeCap) cand[pos] = key;
      }
    }
    __syncthreads();
    cnt = min(k, static_cast<int>(misc[0]));
  }
  // ---- exact order by rank (keys are unique): G threads per candidate ----
  int G = 1;  // a power of two <= 32 with G * cnt <= kMergeThreads, at least 1
  while (G < 32 && 2 * G * cnt <= kMergeThreads) G *= 2;
  const int groups = kMergeThreads / G;
  for (int base = 0; base < cnt; base += groups) {
    const int i = base + tid / G, sub = tid % G;
    const uint64_t key = i < cnt ? cand[i] : 0ull;
    int rank = 0;
    if (i < cnt)
      for (int j = sub; j < cnt; j += G) rank += cand[j] > key;
    for (int o = G / 2; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (i < cnt && sub == 0 && rank < k) put(rank, key);
  }
  for (int r = min(cnt, k) + tid; r < a.k_max; r += kMergeThreads) put(r, 0ull);  // no candidate, and ranks >= k
}

// ---------------------------------------------------------------------------
// One warp per row, for plans whose slots hold at most kWarpItems keys per row
// and lists of at most kWarpMaxK entries (few slots, or short lists: the
// CTA-wide barriers of the kernel above would dominate).  The row's keys are
// held in registers, 16 per lane; the output ranks come out of a tournament:
// every round the warp's largest remaining key (two redux.sync max steps, on
// the high then the low word; keys are unique, so exactly one lane holds it)
// is the next rank, and its holder drops it and recomputes its own best.  k
// rounds, no shared memory and no ranking pass.
// ---------------------------------------------------------------------------
constexpr int kWarpItems = 512;
constexpr int kWarpPerLane = kWarpItems / 32;
constexpr int kWarpMaxK = 32;
constexpr int kWarpRowsPerCtaMax = 8;
constexpr size_t kSlotsSmemMax = 48 * 1024;  // dynamic shared memory of one slots-kernel CTA

__device__ __forceinline__ uint64_t max_of(const uint64_t (&kv)[kWarpPerLane]) {
  uint64_t m = kv[0];
#pragma unroll
  for (int t = 1; t < kWarpPerLane; ++t) m = kv[t] > m ? kv[t] : m;
  return m;
}

// One warp's row: lse = M + log(sum_j s_j exp(m_j - M)) over the row's slots, the
// selected token's logprob, the sampled token (the best slot partial), or in record
// mode the row's record head.  Every lane gets lse.
__device__ __forceinline__ float warp_row_head(const MergeArgs& a, int row, int lane) {
  const int nslots = a.splits;
  const float2* ms = a.parts.part_ms + static_cast<int64_t>(row) * a.splits;
  float tm = -INFINITY, ts = 0.0f;
  for (int j = lane; j < nslots; j += 32) {
    const float2 p = ms[j];
    if (p.x > tm) {
      ts = (tm == -INFINITY) ? 0.0f : ts * expf(tm - p.x);
      tm = p.x;
    }
    if (p.x != -INFINITY) ts += p.y * expf(p.x - tm);
  }
  const float M = warp_max(tm);
  const float S = warp_sum((tm == -INFINITY) ? 0.0f : ts * expf(tm - M));
  const float lse = (M == -INFINITY) ? -INFINITY : M + logf(S);
  if (lane == 0 && a.rec.base != nullptr) {
    write_record_head(a, row, M, S);
  } else if (lane == 0) {
    a.lse[row] = lse;
    if (a.sel) {
      const int t = a.sel[row];
      float v = __int_as_float(0x7fc00000);  // NaN: no selected token / out of range
      if (t >= 0 && t < a.V)
        v = a.parts.sel_logit[row] - lse;
      else if (t != -1)
        set_status(a.dev_status, LMH_DS_SEL_OUT_OF_RANGE);
      a.sel_logprob[row] = v;
    }
  }
  if (a.samp.enabled) {  // the sampled token: the best of the slots' partials
    const float4* ps = a.parts.part_samp + static_cast<int64_t>(row) * a.splits;
    float4 b = make_float4(-INFINITY, __int_as_float(-1), -INFINITY, 0.0f);
    for (int j = lane; j < a.splits; j += 32) {
      const float4 c = ps[j];
      if (samp_better(c, b)) b = c;
    }
    b = samp_warp_best(b);
    if (lane == 0) samp_write(a, row, b, lse);
  }
  return lse;
}

// Writes a warp's ranks: rank r's key comes out of round r (the same key in every
// lane); lane r % 32 keeps it and the lanes store 32 ranks at a time, coalesced.
// Ranks >= k get (-1, -inf), or key 0 in record mode.
struct WarpRankWriter {
  int32_t* ids;
  float* lps;
  unsigned long long* keys;  // record mode
  float lse;
  uint64_t my_key = 0;

  __device__ __forceinline__ WarpRankWriter(const MergeArgs& a, int row, float lse_) : lse(lse_) {
    const bool rec = a.rec.base != nullptr;
    ids = rec ? nullptr : a.topk_ids + static_cast<int64_t>(row) * a.k_max;
    lps = rec ? nullptr : a.topk_logprobs + static_cast<int64_t>(row) * a.k_max;
    keys = rec ? record_keys(row_record(a, row)) : nullptr;
  }
  __device__ __forceinline__ void put(int r, int k, int lane, uint64_t key) {
    if (lane == (r & 31)) my_key = key;  // key 0: fewer than k candidates
    if ((r & 31) == 31 || r == k - 1) {
      const int r0 = r & ~31;
      if (lane <= (r & 31)) {
        if (keys) {
          keys[r0 + lane] = my_key;
        } else {
          ids[r0 + lane] = my_key ? key_id(my_key) : -1;
          lps[r0 + lane] = my_key ? key_value(my_key) - lse : -INFINITY;
        }
      }
    }
  }
  __device__ __forceinline__ void pad(int k, int k_max, int lane) {
    for (int r = k + lane; r < k_max; r += 32) {
      if (keys) {
        keys[r] = 0ull;
      } else {
        ids[r] = -1;
        lps[r] = -INFINITY;
      }
    }
  }
};

// The warp's largest key among every lane's `cand` (keys are unique: one lane holds it).
__device__ __forceinline__ uint64_t warp_max_key(uint64_t cand) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(cand >> 32));
  const uint32_t lo =
      __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(cand >> 32) == hi ? static_cast<uint32_t>(cand) : 0u);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__global__ void __launch_bounds__(kWarpRowsPerCtaMax * 32) merge_partials_warp_kernel(const MergeArgs a) {
  pdl_wait();  // the partials come from the kernel launched just before
  pdl_launch_dependents();  // a following kernel may be scheduled; it waits for this grid before using its results
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int row = blockIdx.x * (blockDim.x >> 5) + w;
  if (row >= a.rows) return;
  const int nslots = a.splits;

  // ---- every independent load first: K and the row's keys ----
  int k = a.k_max;
  if (a.row_k) k = min(max(a.row_k[row], 0), a.k_max);
  const unsigned long long* keys = a.parts.part_keys + static_cast<int64_t>(row) * a.splits * a.k_max;
  // item i = (slot i / k, rank i % k) of the slots' sorted lists; only the first k of a
  // list can reach the row's top k
  const int n_items = nslots * k;
  uint64_t kv[kWarpPerLane];
#pragma unroll
  for (int t = 0; t < kWarpPerLane; ++t) {
    const int i = lane + 32 * t;
    kv[t] = 0;
    if (i < n_items) {
      const int j = i / k;
      kv[t] = keys[static_cast<int64_t>(j) * a.k_max + (i - j * k)];
    }
  }
  const float lse = warp_row_head(a, row, lane);
  if (a.k_max == 0) return;

  // ---- tournament: rank r is the largest key left after ranks 0..r-1 ----
  WarpRankWriter out(a, row, lse);
  uint64_t best = max_of(kv);
  for (int r = 0; r < k; ++r) {
    const uint64_t key = warp_max_key(best);
    if (key != 0ull && best == key) {  // the one holder drops it
#pragma unroll
      for (int t = 0; t < kWarpPerLane; ++t) kv[t] = kv[t] == key ? 0ull : kv[t];
      best = max_of(kv);
    }
    out.put(r, k, lane, key);
  }
  out.pad(k, a.k_max, lane);
}

// ---------------------------------------------------------------------------
// One warp per row for plans with at most 32 * SPL slots: the warp copies the row's
// lists into shared memory (coalesced), and lane l walks the sorted lists of slots
// l, l + 32, ... (SPL of them) with head pointers, holding each list's current and
// next entries in registers.  Round r: the warp's largest head (warp_max_key over each
// lane's best head) is rank r; the lane that holds it moves that list on by one entry
// and fetches the one after.  A round is a few instructions for the warp, where the
// tournament above rescans a lane's 16 items.
// ---------------------------------------------------------------------------
template <int SPL>
__global__ void __launch_bounds__(kWarpRowsPerCtaMax * 32) merge_partials_slots_kernel(const MergeArgs a) {
  extern __shared__ __align__(16) unsigned long long s_lists[];  // per warp: splits * k_max keys
  __shared__ __align__(8) uint64_t s_bar[kWarpRowsPerCtaMax];     // per warp: its bulk copy
  pdl_wait();  // the partials come from the kernel launched just before
  pdl_launch_dependents();  // a following kernel may be scheduled; it waits for this grid before using its results
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int row = blockIdx.x * (blockDim.x >> 5) + w;
  if (row >= a.rows) return;
  int k = a.k_max;
  if (a.row_k) k = min(max(a.row_k[row], 0), a.k_max);
  const int n = a.splits * a.k_max;
  unsigned long long* lists = s_lists + static_cast<int64_t>(w) * n;
  const unsigned long long* src = a.parts.part_keys + static_cast<int64_t>(row) * n;
  // The row's lists are one contiguous block: one bulk copy when it is large (at least 512
  // keys, an even number from a 16-byte aligned address), else asynchronous 8-byte copies
  // (cp.async), all of a lane's in flight at once (cheaper to start for a small block).
  // Either way the warp waits after the row head's loads have gone out too; entries past
  // a list's first k are never read.
  const bool bulk = n >= 512 && (n & 1) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;
  uint64_t* bar = &s_bar[w];
  if (bulk) {
    if (lane == 0) {
      mbar_init(bar, 1);
      mbar_init_fence();
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * 8u);
      bulk_load(lists, src, static_cast<uint32_t>(n) * 8u, bar);
    }
    __syncwarp();
  } else {
    for (int i = lane; i < n; i += 32)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(lists + i)),
                   "l"(__cvta_generic_to_global(src + i))
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  const float lse = warp_row_head(a, row, lane);
  if (bulk) {
    if (!mbar_wait(bar, 0)) {  // (bounded) the copy lands before the warp goes on
      set_status(a.dev_status, LMH_DS_TIMEOUT);
      mbar_wait(bar, 0);
    }
  } else {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  }
  if (a.k_max == 0) return;
  __syncwarp();

  // only the first k entries of a list can reach the row's top k
  int p[SPL];  // entries of each of this lane's lists already ranked
  uint64_t head[SPL], next[SPL];
#pragma unroll
  for (int i = 0; i < SPL; ++i) {
    const bool has = lane + 32 * i < a.splits;
    const unsigned long long* l = lists + (lane + 32 * i) * a.k_max;
    p[i] = 0;
    head[i] = (has && k > 0) ? l[0] : 0ull;
    next[i] = (has && k > 1) ? l[1] : 0ull;
  }
  WarpRankWriter out(a, row, lse);
  for (int r = 0; r < k; ++r) {
    uint64_t best = head[0];
#pragma unroll
    for (int i = 1; i < SPL; ++i) best = max(best, head[i]);
    const uint64_t key = warp_max_key(best);
    if (key != 0ull && best == key) {  // the one holder moves that list on
#pragma unroll
      for (int i = 0; i < SPL; ++i) {
        if (head[i] == key) {
          head[i] = next[i];
          ++p[i];
          next[i] = (p[i] + 1 < k) ? lists[(lane + 32 * i) * a.k_max + p[i] + 1] : 0ull;
        }
      }
    }
    out.put(r, k, lane, key);
  }
  out.pad(k, a.k_max, lane);
}

// ---------------------------------------------------------------------------
// vocabulary-parallel records -> the merge's partials (one slot per part)
// ---------------------------------------------------------------------------
// Thread t of row r copies part t's (m, s) and keys; the part whose share holds
// the selected token provides its logit.
__global__ void __launch_bounds__(128) unpack_records_kernel(const unsigned char* __restrict__ records,
                                                             int num_parts, int rows, int k_max, Partials parts) {
  const int row = blockIdx.x;
  const size_t rb = record_bytes(k_max);
  for (int p = threadIdx.x; p < num_parts; p += blockDim.x) {
    const VocabRecord* r =
        reinterpret_cast<const VocabRecord*>(records + (static_cast<int64_t>(p) * rows + row) * rb);
    const int64_t slot = static_cast<int64_t>(row) * num_parts + p;
    parts.part_ms[slot] = make_float2(r->m, r->s);
    const unsigned long long* keys = reinterpret_cast<const unsigned long long*>(r + 1);
    for (int j = 0; j < k_max; ++j) parts.part_keys[slot * k_max + j] = keys[j];
    if (r->flags & kRecordHasSel) parts.sel_logit[row] = r->sel_logit;
  }
}

cudaError_t launch_unpack_records(const void* records, int num_parts, int rows, int k_max, Partials parts,
                                  cudaStream_t stream) {
  return launch_kernel(unpack_records_kernel, dim3(rows), dim3(128), 0, stream, false,
                       static_cast<const unsigned char*>(records), num_parts, rows, k_max, parts);
}

cudaError_t merge_setup() { return cudaSuccess; }

cudaError_t launch_merge(int rows, int splits, int V, int k_max, Partials parts, const int32_t* sel,
                         const int32_t* row_k, float* lse, float* sel_logprob, int32_t* topk_ids,
                         float* topk_logprobs, uint32_t* dev_status, cudaStream_t stream, bool pdl,
                         const SampleArgs* samp, int num_sms, const RecordOut* rec) {
  MergeArgs a;
  a.rows = rows;
  a.splits = splits;
  a.V = V;
  a.k_max = k_max;
  a.parts = parts;
  a.sel = sel;
  a.row_k = row_k;
  a.lse = lse;
  a.sel_logprob = sel_logprob;
  a.topk_ids = topk_ids;
  a.topk_logprobs = topk_logprobs;
  a.dev_status = dev_status;
  a.samp = samp ? *samp : SampleArgs{};
  a.rec = rec ? *rec : RecordOut{nullptr, 0, 0};
  const int sms = num_sms > 0 ? num_sms : 1;
  if (splits <= 4 * 32 && k_max <= kWarpMaxK) {
    // rows spread over the SMs first, up to 8 per CTA, within 48 KB of lists per CTA
    const size_t per_warp = static_cast<size_t>(splits) * k_max * sizeof(unsigned long long);
    int rpc = 1;
    while (rpc < kWarpRowsPerCtaMax && static_cast<int64_t>(rows) > static_cast<int64_t>(2 * rpc) * sms &&
           (rpc + 1) * per_warp <= kSlotsSmemMax)
      ++rpc;
    const dim3 grid((rows + rpc - 1) / rpc), block(rpc * 32);
    const size_t smem = rpc * per_warp;
    if (splits <= 32) return launch_kernel(merge_partials_slots_kernel<1>, grid, block, smem, stream, pdl, a);
    if (splits <= 64) return launch_kernel(merge_partials_slots_kernel<2>, grid, block, smem, stream, pdl, a);
    return launch_kernel(merge_partials_slots_kernel<4>, grid, block, smem, stream, pdl, a);
  }
  if (static_cast<int64_t>(splits) * k_max <= kWarpItems && k_max <= kWarpMaxK) {
    // rows spread over the SMs first: one warp per CTA while there are SMs to spare
    int rpc = 1;
    while (rpc < kWarpRowsPerCtaMax && static_cast<int64_t>(rows) > static_cast<int64_t>(2 * rpc) * sms) rpc *= 2;
    return launch_kernel(merge_partials_warp_kernel, dim3((rows + rpc - 1) / rpc), dim3(rpc * 32), 0, stream, pdl,
                         a);
  }

  return launch_kernel(merge_partials_kernel, dim3(rows), dim3(kMergeThreads), 0, stream, pdl, a);
}

}  // namespace lmh
