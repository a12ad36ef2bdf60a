// merge_partials.cu -- combine the per-chunk partials of every row (K5).
//
// openinfer issue #719, "Suggested direction": a numerically sound
// multi-stage reduction that returns lse, the selected-token logprob and the
// top-k as an O(k+1) result.  MTPLX PR #532, "Change": logprob = fp32(logit)
// - lse, evaluated only at the survivors and at the scored token; exact ties
// by ascending id.
//
// One CTA per row (see merge_partials_kernel).
#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

constexpr int kMergeThreads = 256;
constexpr int kMergeCap = 1024;  // candidate keys held in shared memory

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

// One CTA per row:
//   lse = M + log(sum_j s_j * exp(m_j - M)) over the row's slots j, with
//         M = max_j m_j (lse = -inf when every logit is -inf);
//   top-k = the k best keys of the union of the slots' sorted top-k lists.
//         Every slot list holds that piece's k best, so the union holds the
//         row's k best.  L = max over slots of their k-th key is a lower
//         bound of the row's k-th key (one slot alone has k keys >= L), so
//         only keys >= L are gathered; they are ordered by rank.
__global__ void __launch_bounds__(kMergeThreads) merge_partials_kernel(const MergeArgs a) {
  __shared__ uint64_t cand[kMergeCap];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t misc[4];
  __shared__ float red[32];
  __shared__ uint64_t red64[32];
  pdl_wait();  // the partials come from the kernel launched just before
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const float2* ms = a.parts.part_ms + static_cast<int64_t>(row) * a.splits;
  int nslots = a.splits;
  if (a.flat_per > 0) {
    const int64_t b0 = static_cast<int64_t>(row) * a.flat_nblk;
    nslots = static_cast<int>((b0 + a.flat_nblk - 1) / a.flat_per - b0 / a.flat_per) + 1;
  }

  // ---- lse ----
  float tm = -INFINITY, ts = 0.0f;
  for (int j = tid; j < nslots; j += kMergeThreads) {
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
    misc[0] = 0;
  }
  if (a.k_max == 0) return;
  int k = a.k_max;
  if (a.row_k) k = min(max(a.row_k[row], 0), a.k_max);
  int32_t* out_ids = a.topk_ids + static_cast<int64_t>(row) * a.k_max;
  float* out_lp = a.topk_logprobs + static_cast<int64_t>(row) * a.k_max;
  if (k == 0) {
    for (int r = tid; r < a.k_max; r += kMergeThreads) {
      out_ids[r] = -1;
      out_lp[r] = -INFINITY;
    }
    return;
  }

  const unsigned long long* keys = a.parts.part_keys + static_cast<int64_t>(row) * a.splits * a.k_max;
  uint64_t lb = 0;  // lower bound of the row's k-th key
  for (int j = tid; j < nslots; j += kMergeThreads) {
    const uint64_t kk = keys[static_cast<int64_t>(j) * a.k_max + (k - 1)];
    lb = kk > lb ? kk : lb;
  }
  lb = block_max_u64(lb, red64);
  // gather every key >= lb: independent loads over all (slot, rank) items
  const int n_items = nslots * k;
  auto in_set = [&](int i, uint64_t* key) -> bool {
    const int j = i / k, r = i - j * k;
    const uint64_t kk = keys[static_cast<int64_t>(j) * a.k_max + r];
    if (kk == 0ull || kk < lb) return false;
    *key = kk;
    return true;
  };
  for (int i = tid; i < n_items; i += kMergeThreads) {
    uint64_t key = 0;
    if (in_set(i, &key)) {
      const uint32_t pos = atomicAdd(&misc[0], 1u);
      if (pos < kMergeCap) cand[pos] = key;
    }
  }
  __syncthreads();
  int cnt = static_cast<int>(misc[0]);
  if (cnt > kMergeCap) {
    // many exact ties: select the k-th key exactly, then keep the k keys at or above it
    int above;
    const uint64_t T64 = cta_radix_select(in_set, n_items, k, 64, hist, misc + 1, &above);
    __syncthreads();
    if (tid == 0) misc[0] = 0;
    __syncthreads();
    for (int i = tid; i < n_items; i += kMergeThreads) {
      uint64_t key = 0;
      if (in_set(i, &key) && key >= T64) {
        const uint32_t pos = atomicAdd(&misc[0], 1u);  // exactly k of them
        if (pos < kMergeCap) cand[pos] = key;
      }
    }
    __syncthreads();
    cnt = min(k, static_cast<int>(misc[0]));
  }
  // exact order by rank (keys are unique)
  for (int t = tid; t < cnt; t += kMergeThreads) {
    const uint64_t key = cand[t];
    int rank = 0;
    for (int j = 0; j < cnt; ++j) rank += cand[j] > key;
    if (rank < k) {
      out_ids[rank] = key_id(key);
      out_lp[rank] = key_value(key) - lse;
    }
  }
  for (int r = min(cnt, k) + tid; r < a.k_max; r += kMergeThreads) {  // ranks without a candidate, and ranks >= k
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
  return launch_kernel(merge_partials_kernel, dim3(rows), dim3(kMergeThreads), 0, stream, pdl, a);
}

}  // namespace lmh
