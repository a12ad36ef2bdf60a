// select_rows.cu -- which rows of a packed batch are sampled (K1).
//
// vllm-metal release v0.4.0.dev20260831, "Summary": decode rows are kept,
// prefill segment j is sampled at cu_seqlens[num_decode + j + 1] - 1, and the
// compacted prefix sums logits_cu_seqlens describe the gathered rows.
// Readings: a decode sequence keeps all its rows; all_rows_mask[s] keeps
// every row of prefill segment s; an empty prefill segment, a decreasing
// cu_seqlens or cu_seqlens[0] != 0 set LMH_DS_BAD_CU_SEQLENS and the
// offending sequence contributes no row.
//
// One CTA of 1024 threads walks the sequences 1024 at a time: each thread
// counts the rows of one sequence, a block scan turns counts into output
// offsets, and the CTA writes the row indices of the whole group
// cooperatively (so a 1024-row prompt-scoring segment is written by 1024
// threads, not one).
#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

constexpr int kSelectThreads = 1024;

__global__ void __launch_bounds__(kSelectThreads)
    select_rows_kernel(const int32_t* __restrict__ cu, int num_seqs, int num_decode,
                       const uint8_t* __restrict__ mask, int max_out, int32_t* __restrict__ row_idx,
                       int32_t* __restrict__ logits_cu, uint32_t* dev_status) {
  // Launched with programmatic dependent launch: wait for the preceding
  // kernel (which may write cu_seqlens or still read row_idx), then let the
  // gather that follows be scheduled.
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int32_t s_excl[kSelectThreads];
  __shared__ int32_t s_first[kSelectThreads];
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_total;
  __shared__ uint32_t s_bits;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_bits = 0;
    logits_cu[0] = 0;
    if (num_seqs > 0 && cu[0] != 0) s_bits |= LMH_DS_BAD_CU_SEQLENS;
  }
  int64_t running = 0;  // rows selected by earlier groups (same value in every thread)
  for (int base = 0; base < num_seqs; base += kSelectThreads) {
    const int s = base + tid;
    int cnt = 0, first = 0;
    if (s < num_seqs) {
      const int lo = cu[s], hi = cu[s + 1];
      const bool every = (s < num_decode) || (mask != nullptr && mask[s] != 0);
      if (hi < lo) {
        atomicOr(&s_bits, LMH_DS_BAD_CU_SEQLENS);
      } else if (every) {
        first = lo;
        cnt = hi - lo;
      } else if (hi == lo) {
        atomicOr(&s_bits, LMH_DS_BAD_CU_SEQLENS);
      } else {
        first = hi - 1;
        cnt = 1;
      }
    }
    // block-wide exclusive scan of cnt
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = s_warp[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += t;
      }
      s_warp[lane] = wi - w;  // exclusive prefix of the warp totals
      if (lane == 31) s_total = wi;
    }
    __syncthreads();
    const int excl = incl - cnt + s_warp[warp];
    s_excl[tid] = excl;
    s_first[tid] = first;
    if (s < num_seqs) logits_cu[s + 1] = static_cast<int32_t>(running + excl + cnt);
    __syncthreads();
    const int total = s_total;
    const int group = min(kSelectThreads, num_seqs - base);
    // write the group's rows: output slot r belongs to the last sequence whose offset is <= r
    for (int r = tid; r < total; r += kSelectThreads) {
      int lo = 0, hi = group - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_excl[mid] <= r)
          lo = mid;
        else
          hi = mid - 1;
      }
      const int64_t slot = running + r;
      if (slot < max_out)
        row_idx[slot] = s_first[lo] + (r - s_excl[lo]);
      else
        atomicOr(&s_bits, LMH_DS_ROWS_OVERFLOW);
    }
    running += total;
    __syncthreads();
  }
  __syncthreads();
  if (tid == 0 && s_bits) set_status(dev_status, s_bits);
}

cudaError_t launch_select_rows(const int32_t* cu, int num_seqs, int num_decode, const uint8_t* mask,
                               int max_out, int32_t* row_idx, int32_t* logits_cu, uint32_t* dev_status,
                               cudaStream_t stream) {
  return launch_kernel(select_rows_kernel, dim3(1), dim3(kSelectThreads), 0, stream, true, cu, num_seqs, num_decode,
                       mask, max_out, row_idx, logits_cu, dev_status);
}

}  // namespace lmh
