// device_common.cuh -- device helpers shared by the liblmh kernels (sm_103a).
//
// * Sortable keys.  A candidate (logit v, token id) is packed into one 64-bit
//   key whose unsigned order is the output order of the top-k: larger logit
//   first, exact ties by ascending id (MTPLX PR #532, "Change").  Keys are
//   unique per id; the value 0 never occurs for a real entry and marks an
//   empty slot.
// * Bounded mbarrier waits (every spin has a time limit and reports
//   LMH_DS_TIMEOUT instead of hanging).
// * CTA-wide reductions, a radix select of the k-th largest key and a
//   bitonic sort of keys in shared memory.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "lmh.h"

namespace lmh {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait

// ---------------------------------------------------------------------------
// keys
// ---------------------------------------------------------------------------

// Order-preserving map of an fp32 value to uint32 (-0.0 folded into +0.0 so
// that the two compare as the exact tie they are).
__device__ __forceinline__ uint32_t f32_ord(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ord_f32(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t make_key(float v, int32_t id) {
  return (static_cast<uint64_t>(f32_ord(v)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(id));
}

__device__ __forceinline__ float key_value(uint64_t key) {
  return ord_f32(static_cast<uint32_t>(key >> 32));
}

__device__ __forceinline__ int32_t key_id(uint64_t key) {
  return static_cast<int32_t>(~static_cast<uint32_t>(key));
}

// ---------------------------------------------------------------------------
// status + timers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void set_status(uint32_t* dev_status, uint32_t bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers, bulk copies
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make initialised barriers visible to the async proxy (TMA, tensor cores).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs and returns false (the caller reports LMH_DS_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Non-blocking test of a phase's completion (mbarrier.test_wait).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Limits below this are test settings (lmh_debug_set_wait_limit): such a wait
// polls with test_wait, because try_wait itself may suspend the thread until
// the phase completes and so outlast a limit shorter than its own window.
constexpr uint64_t kPollLimitNs = 1000000ull;

// Wait on an mbarrier unless the CTA has aborted (another thread gave up
// first); after limit_ns, mark the abort and report LMH_DS_TIMEOUT.  The
// kernels pass the library's wait limit (2 s unless a test shortened it);
// the waits that drain a CTA's copies in flight after an abort use mbar_wait
// and keep the full limit.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* dev_status, uint64_t limit_ns = kWaitLimitNs) {
  const bool poll = limit_ns < kPollLimitNs;
  if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!(poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      set_status(dev_status, LMH_DS_TIMEOUT);
      return false;
    }
  }
  return true;
}

// One-dimensional bulk copy global -> shared, completing on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read once: its lines are evicted first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy for data read again soon: its lines are evicted last.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// fp32 store with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void st_keep(float* dst, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(dst), "f"(v), "l"(policy) : "memory");
}

// bulk_load with an L2 cache policy (from createpolicy).
__device__ __forceinline__ void bulk_load_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// A kernel launched with the programmatic-serialization attribute may start
// while its predecessor in the stream is still running; pdl_wait() blocks
// until the predecessor has completed and its writes are visible (a no-op
// without such a predecessor).  pdl_launch_dependents() lets the successor be
// scheduled once every CTA of this grid has executed it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// CTA-wide max / sum; `scratch` holds >= 32 floats; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = (lane < nw) ? scratch[lane] : -INFINITY;
  r = warp_max(r);
  return r;
}

__device__ __forceinline__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = (lane < nw) ? scratch[lane] : 0.0f;
  r = warp_sum(r);
  return r;
}

__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  uint64_t r = (lane < nw) ? scratch[lane] : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t w = __shfl_xor_sync(0xffffffffu, r, o);
    r = w > r ? w : r;
  }
  return r;
}

// 2^x on the special-function unit (PTX ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// named barriers (a subset of a CTA's warps synchronising among themselves)
// ---------------------------------------------------------------------------
// bar.sync / bar.red on barrier `id` for `n` threads (n a multiple of 32; every
// thread of the participating warps arrives).  Barrier 0 is __syncthreads'.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier that also returns the OR of every participating thread's `pred`.
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------------------
// radix select: the k-th largest 64-bit key of an item set
// ---------------------------------------------------------------------------
//
// Items are enumerated by index 0..n-1 through `get(i, &key)`, which returns
// false for items that are not in the set.  Only the top `bits` bits of the
// keys take part (bits a multiple of 8, <= 64).  Returns the prefix T (in the
// top `bits` bits, lower bits 0) of the k-th largest key and writes to
// *n_above the number of set items whose prefix is strictly greater than T
// (< k); items with prefix == T fill the ranks n_above..k-1 (and maybe more).
// With bits = 64 and unique keys exactly k items have key >= T.
// Requires k >= 1 and at least k items in the set.  `hist` is 256 uint32 of
// shared memory, `bcast` 2 uint32 of shared memory.  Run by a group of `nt`
// threads (whole warps) with ranks tid = 0..nt-1, synchronised by `sync()`.
template <typename Get, typename Sync>
__device__ uint64_t group_radix_select(Get get, int n, int k, int bits, uint32_t* hist, uint32_t* bcast,
                                       int* n_above, int tid, int nt, Sync sync) {
  uint64_t prefix = 0, mask = 0;
  int need = k, above = 0;
  for (int shift = 56; shift >= 64 - bits; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    sync();
    for (int base = 0; base < n; base += nt) {
      const int i = base + tid;
      uint64_t key = 0;
      bool in = (i < n) && get(i, &key) && ((key & mask) == prefix);
      const uint32_t digit = in ? static_cast<uint32_t>(key >> shift) & 0xFFu : 0x100u;
      // warp-aggregated increment: one atomic per distinct digit in the warp
      const unsigned active = __ballot_sync(0xffffffffu, in);
      if (in) {
        const unsigned peers = __match_any_sync(active, digit);
        if ((tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    sync();
    if (tid < 32) {
      // find digit d with count(> d) < need <= count(>= d), scanning from 255 down
      const int lane = tid;
      uint32_t c[8];
      uint32_t mine = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - (lane * 8 + j)];
        mine += c[j];
      }
      // inclusive prefix over lanes (lane 0 holds the largest digits)
      uint32_t incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t excl = incl - mine;
      const bool hit = excl < static_cast<uint32_t>(need) && incl >= static_cast<uint32_t>(need);
      if (hit) {
        uint32_t run = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= static_cast<uint32_t>(need)) {
            bcast[0] = 255 - (lane * 8 + j);
            bcast[1] = run;
            break;
          }
          run += c[j];
        }
      }
    }
    sync();
    const uint32_t d = bcast[0];
    const uint32_t gt = bcast[1];
    sync();
    need -= static_cast<int>(gt);
    above += static_cast<int>(gt);
    prefix |= static_cast<uint64_t>(d) << shift;
    mask |= 0xFFull << shift;
  }
  *n_above = above;
  return prefix;
}

// The same over all threads of the CTA (synchronised by __syncthreads).
template <typename Get>
__device__ uint64_t cta_radix_select(Get get, int n, int k, int bits, uint32_t* hist, uint32_t* bcast,
                                     int* n_above) {
  return group_radix_select(get, n, k, bits, hist, bcast, n_above, static_cast<int>(threadIdx.x),
                            static_cast<int>(blockDim.x), [] { __syncthreads(); });
}

// ---------------------------------------------------------------------------
// bitonic sort of keys in shared memory, descending
// ---------------------------------------------------------------------------
// keys[0..n) with n a power of two (pad with 0 = empty).  All threads call it.
__device__ __forceinline__ void cta_bitonic_sort_desc(uint64_t* keys, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int t = threadIdx.x; t < (n >> 1); t += blockDim.x) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const uint64_t a = keys[lo], b = keys[hi];
        if ((a < b) == desc) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
    }
  }
  __syncthreads();
}

__host__ __device__ constexpr int next_pow2(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

}  // namespace lmh
