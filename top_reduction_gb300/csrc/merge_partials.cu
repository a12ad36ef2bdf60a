// merge_partials.cu -- combine the per-chunk partials of every row (K5).
//
// openinfer issue #719, "Suggested direction": a numerically sound
// multi-stage reduction that returns lse, the selected-token logprob and the
// top-k as an O(k+1) result.  MTPLX PR #532, "Change": logprob = fp32(logit)
// - lse, evaluated only at the survivors and at the scored token; exact ties
// by ascending id.
//
// One warp per row, warp-level primitives only (see merge_partials_kernel).
#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

constexpr int kMergeWarps = 8;      // rows per CTA: one warp per row
constexpr int kMergeWarpCap = 256;  // candidate keys per warp held in shared memory

struct MergeArgs {
  int rows, splits, V, k_max;
  int flat_per, flat_nblk;  // flat_per > 0: the slots a row fills follow the range layout
  Partials parts;
  const int32_t* sel;
  const int32_t* row_k;
  float* lse;
  float* sel_logprob;
  int32_t* topk_ids;
  float* topk_logprobs;
  uint32_t* dev_status;
};

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Warp-level radix select: the k-th largest of the keys get(i) (i < n) that are
// in the set; all 64 bits take part, so exactly k set items have key >= the
// result (keys are unique).  `hist` is 256 uint32 of this warp's shared memory.
template <typename Get>
__device__ uint64_t warp_radix_select(Get get, int n, int k, uint32_t* hist) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0, mask = 0;
  int need = k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      uint64_t key = 0;
      const bool in = i < n && get(i, &key) && (key & mask) == prefix;
      const unsigned active = __ballot_sync(0xffffffffu, in);
      if (in) {
        const uint32_t digit = static_cast<uint32_t>(key >> shift) & 0xFFu;
        const unsigned peers = __match_any_sync(active, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    __syncwarp();
    uint32_t c[8], mine = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c[j] = hist[255 - (lane * 8 + j)];
      mine += c[j];
    }
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - mine;
    uint32_t found = 0xFFFFFFFFu, gt = 0;
    if (excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need)) {
      uint32_t run = excl;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (found == 0xFFFFFFFFu && run + c[j] >= static_cast<uint32_t>(need)) {
          found = 255 - (lane * 8 + j);
          gt = run;
        }
        run += c[j];
      }
    }
    const unsigned who = __ballot_sync(0xffffffffu, found != 0xFFFFFFFFu);
    const int src = __ffs(who) - 1;
    const uint32_t d = __shfl_sync(0xffffffffu, found, src);
    gt = __shfl_sync(0xffffffffu, gt, src);
    need -= static_cast<int>(gt);
    prefix |= static_cast<uint64_t>(d) << shift;
    mask |= 0xFFull << shift;
  }
  return prefix;
}

// One warp per row:
//   lse = M + log(sum_j s_j * exp(m_j - M)) over the row's slots j, with
//         M = max_j m_j (lse = -inf when every logit is -inf);
//   top-k = the k best keys of the union of the slots' sorted top-k lists.
//         Every slot list holds that piece's k best, so the union holds the
//         row's k best.  L = max over slots of their k-th key is a lower
//         bound of the row's k-th key (one slot alone has k keys >= L), so
//         only keys >= L are gathered; their order comes from their ranks.
__global__ void __launch_bounds__(kMergeWarps * 32) merge_partials_kernel(const MergeArgs a) {
  __shared__ uint64_t cand_all[kMergeWarps][kMergeWarpCap];
  __shared__ uint32_t hist_all[kMergeWarps][256];
  pdl_wait();  // the partials come from the kernel launched just before
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kMergeWarps + warp;
  if (row >= a.rows) return;  // whole warps only: nothing below synchronises the CTA
  uint64_t* cand = cand_all[warp];

  const float2* ms = a.parts.part_ms + static_cast<int64_t>(row) * a.splits;
  int nslots = a.splits;
  if (a.flat_per > 0) {
    const int64_t b0 = static_cast<int64_t>(row) * a.flat_nblk;
    nslots = static_cast<int>((b0 + a.flat_nblk - 1) / a.flat_per - b0 / a.flat_per) + 1;
  }

  // ---- lse ----
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

  if (lane == 0) {
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
  if (a.k_max == 0) return;

  int k = a.k_max;
  if (a.row_k) k = min(max(a.row_k[row], 0), a.k_max);
  int32_t* out_ids = a.topk_ids + static_cast<int64_t>(row) * a.k_max;
  float* out_lp = a.topk_logprobs + static_cast<int64_t>(row) * a.k_max;
  if (k == 0) {
    for (int r = lane; r < a.k_max; r += 32) {
      out_ids[r] = -1;
      out_lp[r] = -INFINITY;
    }
    return;
  }

  const unsigned long long* keys = a.parts.part_keys + static_cast<int64_t>(row) * a.splits * a.k_max;
  uint64_t lb = 0;  // lower bound of the row's k-th key
  for (int j = lane; j < nslots; j += 32) {
    const uint64_t kk = keys[static_cast<int64_t>(j) * a.k_max + (k - 1)];
    lb = kk > lb ? kk : lb;
  }
  lb = warp_max_u64(lb);

  const int n_items = nslots * k;
  auto in_set = [&](int i, uint64_t* key) -> bool {
    const int j = i / k, r = i - j * k;
    const uint64_t kk = keys[static_cast<int64_t>(j) * a.k_max + r];
    if (kk == 0ull || kk < lb) return false;
    *key = kk;
    return true;
  };
  int count = 0;
  for (int base = 0; base < n_items; base += 32) {
    uint64_t key = 0;
    const bool in = (base + lane) < n_items && in_set(base + lane, &key);
    const unsigned bal = __ballot_sync(0xffffffffu, in);
    const int pos = count + __popc(bal & ((1u << lane) - 1u));
    if (in && pos < kMergeWarpCap) cand[pos] = key;
    count += __popc(bal);
  }
  if (count > kMergeWarpCap) {
    // many exact ties: select the k-th key exactly, then keep the k keys at or above it
    const uint64_t T64 = warp_radix_select(in_set, n_items, k, hist_all[warp]);
    count = 0;
    for (int base = 0; base < n_items; base += 32) {
      uint64_t key = 0;
      const bool in = (base + lane) < n_items && in_set(base + lane, &key) && key >= T64;
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      const int pos = count + __popc(bal & ((1u << lane) - 1u));
      if (in && pos < kMergeWarpCap) cand[pos] = key;
      count += __popc(bal);
    }
    count = min(count, k);
  }
  __syncwarp();
  // exact order by rank (keys are unique)
  for (int t = lane; t < count; t += 32) {
    const uint64_t key = cand[t];
    int rank = 0;
    for (int j = 0; j < count; ++j) rank += cand[j] > key;
    if (rank < k) {
      out_ids[rank] = key_id(key);
      out_lp[rank] = key_value(key) - lse;
    }
  }
  for (int r = count + lane; r < a.k_max; r += 32) {
    out_ids[r] = -1;
    out_lp[r] = -INFINITY;
  }
}

cudaError_t merge_setup() { return cudaSuccess; }

cudaError_t launch_merge(int rows, int splits, int V, int k_max, Partials parts, const int32_t* sel,
                         const int32_t* row_k, float* lse, float* sel_logprob, int32_t* topk_ids,
                         float* topk_logprobs, uint32_t* dev_status, cudaStream_t stream, int flat_per,
                         int flat_nblk, bool pdl) {
  MergeArgs a;
  a.flat_per = flat_per;
  a.flat_nblk = flat_nblk;
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
  return launch_kernel(merge_partials_kernel, dim3((rows + kMergeWarps - 1) / kMergeWarps), dim3(kMergeWarps * 32), 0,
                       stream, pdl, a);
}

}  // namespace lmh
