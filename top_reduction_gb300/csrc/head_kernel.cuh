// head_kernel.cuh -- the tcgen05 head kernel (K3) with its fused per-row
// reduction, shared by the translation units that instantiate it (one per
// sampling mode, compiled in parallel) and by the host code in head_gemm.cu.
//
// GB300 design (sm_103a):
//   * D[128 rows x 256 vocab] tiles, z = A . W^T with A = gathered hidden rows
//     [rows x H] and W = lm_head.weight [V x H]; both operands are K-major.
//   * warp 0: TMA producer.  64-element (128-byte) slices of A and W are
//     loaded with cp.async.bulk.tensor into a ring of shared-memory stages
//     using the 128-byte swizzle, completing on "full" mbarriers.
//   * warp 1: allocates 512 TMEM columns (two 256-column fp32 accumulators)
//     and one thread issues tcgen05.mma (kind::f16, bf16 in, fp32 out in
//     TMEM); tcgen05.commit frees a stage ("empty") once its MMAs have read
//     it and signals an accumulator ("acc_full") when a tile is complete.
//   * warps 2..5: epilogue.  Warp w reads TMEM lanes 32*(w%4)..+31, so each
//     thread owns one row.  Per 64-column block it keeps the running max m
//     and sum exp(z - m) (online rescaling), the block maximum, and inserts
//     into the row's sorted top-k list only the entries of blocks whose
//     maximum exceeds the current k-th value tau (the block-max prefilter
//     applied while streaming; ids ascend within a CTA's range, so an equal
//     value never displaces an earlier id).  It also captures z[row][sel].
//   * Persistent CTAs walk "units" = (128-row tile, vocabulary range); the
//     per-row state lives across the n-tiles of a unit and is flushed as one
//     partial per (row, range) that merge_partials.cu combines.
//   * Batches of at most 64 rows with a heavy epilogue (sampling, or longer
//     lists on short tiles) split each tile's columns over the four epilogue
//     warps: the A stage holds a copy of the rows in every lane quarter that
//     the warps then share out (HeadArgs::rep).  Batches of at most 32 rows
//     with a light epilogue take the deep layout instead (HeadCfg<KCAP, true>):
//     small A slices and 6 stages, so more of W is in flight.
//   * An epilogue warp hands the accumulator back to the MMA as soon as its
//     last block of the tile is in registers.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "lmh_internal.h"

namespace lmh {

constexpr int kBM = 128;    // rows per tile = TMEM lanes
constexpr int kBN = 256;    // vocabulary columns per tile = fp32 TMEM columns per accumulator
constexpr int kBK = 64;     // hidden elements per stage: one 128-byte swizzle row
constexpr int kUmmaK = 16;  // K of one tcgen05.mma kind::f16
constexpr int kHeadThreads = 192;
constexpr int kTmemCols = 512;
constexpr uint32_t kStageBytesA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kStageBytesB = kBN * kBK * 2;  // 32 KB
// W slices the producer prefetches into L2 past its ring while it waits for the kernel
// before it (the grid-dependency wait): HBM keeps streaming W during that wait instead of
// idling once the ring is full.  Prefetching in the steady state measured slower.
constexpr int kWaitPrefetch = 16;

// KCAP: per-row candidate capacity.  KCAP <= 32 keeps each row's top-k list
// in registers and uses the shared region to stage candidate blocks (4 warps x
// 64 columns x 32 lanes x 4 bytes); KCAP 128 keeps a min-heap per row in
// shared memory (slot-major) and has room for only 2 pipeline stages.
//
// kDeep: the layout of batches of at most 32 rows whose epilogue is one warp (no column
// split): A slices of 32 rows (4 KB; the MMA still reads 128 rows from a slice's base, and
// the rows past it only reach accumulator lanes no warp reads), one warp's staging region,
// and 6 stages in place of 4, so more of W is in flight.
template <int KCAP, bool kDeep = false>
struct HeadCfg {
  static constexpr bool kRegList = KCAP <= 32;
  static constexpr int kStages = kDeep ? 6 : (kRegList ? 4 : 2);
  static constexpr uint32_t kStageA = kDeep ? 32 * kBK * 2 : kStageBytesA;
  static constexpr size_t kListBytes = kDeep ? static_cast<size_t>(64) * 32 * 4
                                       : kRegList ? static_cast<size_t>(4) * 64 * 32 * 4
                                                  : static_cast<size_t>(kBM) * KCAP * 8;
  // Small batches may split each tile's columns over the epilogue warps (see
  // HeadArgs::rep); a warp then hands its row state to the leader through its
  // own staging region: 7 words plus (value, id) per list entry, per lane.
  static constexpr bool kRepOk = kRegList && 7 + 2 * KCAP <= 64;
  // column split: every copy's current list threshold, one (unit, value) word per lane
  static constexpr size_t kTauBytes = kRepOk ? 4 * 32 * 8 : 0;
  static constexpr size_t kSmem = 1024 /*alignment slack*/ + kStages * (kStageA + kStageBytesB) +
                                  kListBytes + (2 * kStages + 7) * 8 + 16 + kTauBytes;
};

struct HeadArgs {
  uint32_t a_bytes;  // bytes one A box brings per stage (rows of the box x 128)
  int rows, H, V, k_max;
  int m_tiles, n_tiles, splits, tiles_per_split, num_units;
  const int32_t* sel;
  const int32_t* row_k;
  Partials parts;
  float* logits_out;
  uint32_t* dev_status;
  int epi_quarters;  // TMEM lane quarters that ever hold rows: ceil(rows / 32) below 128 rows, else 4
  // Column split for batches of at most 64 rows: the A stage holds `rep`
  // copies of the rows, each spanning rep_nq lane quarters, so every lane
  // quarter has the rows and epilogue warp q (copy q / rep_nq) reduces only
  // the 64-column blocks c == copy (mod rep) of each tile.  rep 1: off.
  int rep, rep_nq;
  float logit_scale;  // head transform: every logit is logit_scale * (A . W) (1: none)
  SampleArgs samp;    // device-side sampling (kernels with kSamp != 0)
  int final_out;   // one vocabulary split: write the final results (out), not partials
  RowOutputs out;
  uint64_t wait_ns;  // limit of a bounded wait on another role of the CTA
  int id_off;  // vocabulary-parallel share: token id of W's first row (0: the whole head)
};

// ---------------------------------------------------------------------------
// PTX wrappers: TMA, tcgen05
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// Bulk tensor prefetch of one box into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), descriptor
// version 1, leading byte offset unused for this layout (set to 16 bytes).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(16u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared-memory matrix descriptor: vocabulary-major (MN-major) W slice of a
// [H x V] head, 128-byte swizzle.  The slice is 4 blocks of 64 vocabulary
// columns (128-byte rows) x 64 hidden rows, 8 KB apart; within a block, groups
// of 8 hidden rows are 1024 bytes apart.  One MMA reads 16 hidden rows: its
// start address advances by 2048 bytes per K step.
constexpr uint32_t kHvBlockBytes = 64 * kBK * 2;  // 8 KB: 64 vocabulary columns x 64 hidden rows
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(kHvBlockBytes >> 4) << 16;  // between 64-column blocks (MN direction)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;          // between 8-row groups (K direction)
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major (kIdesc) or MN-major (kIdescBmn, bit 16), N = kBN, M = kBM.
constexpr uint32_t kIdesc = (1u << 4)                                   // D format: f32
                            | (1u << 7)                                 // A format: bf16
                            | (1u << 10)                                // B format: bf16
                            | (static_cast<uint32_t>(kBN >> 3) << 17)   // N / 8
                            | (static_cast<uint32_t>(kBM >> 4) << 24);  // M / 16
constexpr uint32_t kIdescBmn = kIdesc | (1u << 16);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate,
                                          uint32_t idesc = kIdesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Load 64 consecutive fp32 columns of this thread's TMEM lane and wait for
// them in the same asm statement, so no use of the registers can be scheduled
// before tcgen05.wait::ld.  Warp-collective: the whole warp must be converged.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// per-row top-k heap in shared memory (KCAP 128; slot-major: heap[i*128+r])
// ---------------------------------------------------------------------------
// A min-heap of keys: the root is the worst held entry, so tau (the value a
// new entry must exceed once kh entries are held) is the root's value, and an
// insertion costs O(log kh) steps whatever the new entry's rank.  The heap is
// sorted once, at the end of a unit.
struct HeapState {
  float tau;  // value of the root once the heap holds kh keys, else -inf
  int cnt;
};

static __device__ __noinline__ HeapState heap_push(uint64_t* h, int r, HeapState st, int kh, uint64_t key) {
  int i;
  if (st.cnt < kh) {  // grow: sift up from the new last slot
    i = st.cnt++;
    while (i > 0) {
      const int p = (i - 1) >> 1;
      const uint64_t pk = h[p * kBM + r];
      if (pk <= key) break;
      h[i * kBM + r] = pk;
      i = p;
    }
  } else {  // full (the caller only pushes keys above the root): replace the root, sift down
    i = 0;
    for (;;) {
      const int l = 2 * i + 1;
      if (l >= kh) break;
      uint64_t ck = h[l * kBM + r];
      int c = l;
      if (l + 1 < kh) {
        const uint64_t rk = h[(l + 1) * kBM + r];
        if (rk < ck) {
          ck = rk;
          c = l + 1;
        }
      }
      if (ck >= key) break;
      h[i * kBM + r] = ck;
      i = c;
    }
  }
  h[i * kBM + r] = key;
  st.tau = (st.cnt == kh) ? key_value(h[r]) : -INFINITY;
  return st;
}

// Heapsort of the n held keys into descending order (best first): the root
// (the minimum) moves to the end of the shrinking heap.
static __device__ __noinline__ void heap_sort_desc(uint64_t* h, int r, int n) {
  for (int end = n - 1; end > 0; --end) {
    const uint64_t top = h[r];
    const uint64_t key = h[end * kBM + r];
    h[end * kBM + r] = top;
    int i = 0;
    for (;;) {
      const int l = 2 * i + 1;
      if (l >= end) break;
      uint64_t ck = h[l * kBM + r];
      int c = l;
      if (l + 1 < end) {
        const uint64_t rk = h[(l + 1) * kBM + r];
        if (rk < ck) {
          ck = rk;
          c = l + 1;
        }
      }
      if (ck >= key) break;
      h[i * kBM + r] = ck;
      i = c;
    }
    h[i * kBM + r] = key;
  }
}

// ---------------------------------------------------------------------------
// per-row top-k list in registers (KCAP <= 32)
// ---------------------------------------------------------------------------
// The largest float below x (x itself for -inf and NaN).
__device__ __forceinline__ float float_below(float x) {
  if (!(x > -INFINITY)) return x;
  if (x == 0.0f) return -1.40129846e-45f;  // the negative denormal nearest zero
  const uint32_t b = __float_as_uint(x);
  return __uint_as_float(x > 0.0f ? b - 1u : b + 1u);
}

// V[0..KC) holds the row's best values sorted descending, I[] their ids
// (-inf / -1 in empty slots).  Entries reach a thread with ascending ids (the
// tiles of a unit, the blocks of a tile and the columns of a block are
// visited in order), so a new entry ranks after every held entry of equal
// value and the list stays ordered by (value desc, id asc) with value
// comparisons alone.  Insertion is a branchless shift: slot i keeps its entry
// if it is >= x, takes x if it is the first slot below x, otherwise takes
// slot i-1's entry.  tau = V[KC-1]: only values strictly above it can still
// enter.  The list keeps KC >= k entries; a row reads its first k.
template <int KC>
struct RegTopK {
  float V[KC];
  int32_t I[KC];
  float tau;

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      V[i] = -INFINITY;
      I[i] = -1;
    }
    tau = -INFINITY;
  }

  __device__ __forceinline__ void insert(float x, int32_t id) {
    bool ge[KC];
#pragma unroll
    for (int i = 0; i < KC; ++i) ge[i] = V[i] >= x;
#pragma unroll
    for (int i = KC - 1; i >= 0; --i) {
      const bool prev_ge = (i == 0) || ge[i > 0 ? i - 1 : 0];
      const float pv = V[i > 0 ? i - 1 : 0];
      const int32_t pi = I[i > 0 ? i - 1 : 0];
      V[i] = ge[i] ? V[i] : (prev_ge ? x : pv);
      I[i] = ge[i] ? I[i] : (prev_ge ? id : pi);
    }
    tau = V[KC - 1];
  }

  // sortable key of slot j (0 for an empty slot)
  __device__ __forceinline__ uint64_t key(int j) const { return I[j] >= 0 ? make_key(V[j], I[j]) : 0ull; }
};

// ---------------------------------------------------------------------------
// Gumbel-max sampling noise
// ---------------------------------------------------------------------------
// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): per round two 32x32->64 products
// of counter words with the round multipliers; the high halves are XORed
// with the other counter words and the key; the key grows by the Weyl
// increments.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

// Gumbel noise g = -log(E), E = -log u, of one Philox word, u = ((w >> 9) + 0.5) * 2^-23
// (exact in fp32, strictly inside (0, 1)).  u <= 1 - 2^-24 bounds the noise:
// g <= -log(-log(1 - 2^-24)) < kGumbelMax.  Large g comes from u near 1, where the fast
// logarithm's absolute error would be large relative to log u; there (r = 1 - u < 1/16,
// exact in fp32) E is the Taylor series -log(1 - r) = r + r^2/2 + ... + r^7/7, whose
// truncation is below 2^-29 relative.  Elsewhere |log u| > 1/16 and the fast logarithm's
// error stays below 1e-5 relative, as does that of the outer logarithm on g.
constexpr float kGumbelMax = 16.65f;
__device__ __forceinline__ float exp_variate(uint32_t w) {
  const uint32_t k = w >> 9;
  const float r = (static_cast<float>(0x800000u - k) - 0.5f) * 1.1920928955078125e-7f;
  float p = fmaf(r, 1.0f / 7.0f, 1.0f / 6.0f);
  p = fmaf(r, p, 0.2f);
  p = fmaf(r, p, 0.25f);
  p = fmaf(r, p, 1.0f / 3.0f);
  p = fmaf(r, p, 0.5f);
  p = fmaf(r, p, 1.0f);
  const float e_log = -__logf((static_cast<float>(k) + 0.5f) * 1.1920928955078125e-7f);
  return r < 0.0625f ? r * p : e_log;
}
__device__ __forceinline__ float gumbel_of(uint32_t w) { return -__logf(exp_variate(w)); }

// Candidate test on the raw word: with E >= 1 - u, a token can reach noise above t only
// if 2^23 (1 - u) + 0.5 = 2^23 - (w >> 9) < 2^23 e^-t + 1.  The bound is rounded up (by
// 1e-3 relative and two units, far above the fp32 error of t and of the noise), so the
// words it rejects are words whose noise cannot lift the token above the row's best.
__device__ __forceinline__ uint32_t noise_word_limit(float t) {
  const float thr = __expf(-t) * 8396996.608f + 2.0f;  // 2^23 * 1.001
  return thr < 16777216.0f ? static_cast<uint32_t>(thr) : 0xFFFFFFFFu;  // NaN / inf: every word
}

// ---------------------------------------------------------------------------
// the fused kernel
// ---------------------------------------------------------------------------
// kSamp: 0 no sampling; 1 and 2 draw a token per row, scoring every token of a block
// (kSampAll) or only the tokens whose Philox word passes the candidate test (kSampFiltered).
constexpr int kSampNone = 0, kSampAll = 1, kSampFiltered = 2;

// kHV: W stored [H x V] (vocabulary contiguous): 4 boxes of 64 columns per W slice and a
// vocabulary-major (MN-major) MMA operand.
template <int KCAP, bool kMaterialize, int kSamp, bool kDeep = false, bool kHV = false>
__global__ void __launch_bounds__(kHeadThreads, 1)
    head_logprobs_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const HeadArgs a) {
  using Cfg = HeadCfg<KCAP, kDeep>;
  static_assert(!kDeep || (Cfg::kRegList && kSamp == 0), "the deep layout: register lists, no sampling");
  constexpr int S = Cfg::kStages;
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned (the 128-B swizzle atoms), as an offset from smem_raw so that the
  // compiler still sees shared-memory pointers (plain LDS/STS, not generic accesses)
  unsigned char* smem =
      smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
  unsigned char* sA = smem;
  unsigned char* sB = sA + S * Cfg::kStageA;
  uint64_t* lists = reinterpret_cast<uint64_t*>(sB + S * kStageBytesB);
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<unsigned char*>(lists) + Cfg::kListBytes);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* xchg_full = acc_empty + 2;    // column split: the copies' row states are staged
  uint64_t* xchg_empty = xchg_full + 1;   // column split: the leader has read them
  uint64_t* mma_drain = xchg_empty + 1;   // the MMA thread's work in flight has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // column split: [lane quarter][lane] (unit << 32 | threshold bits) of each row copy
  volatile uint64_t* tau_sh =
      reinterpret_cast<volatile uint64_t*>(reinterpret_cast<unsigned char*>(full) + (2 * S + 7) * 8 + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k_blocks = (a.H + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], a.epi_quarters * 32);  // the epilogue warps that read accumulators
    }
    mbar_init(xchg_full, a.rep > 1 ? (4 - a.rep_nq) * 32 : 1);
    mbar_init(xchg_empty, a.rep > 1 ? a.rep_nq * 32 : 1);
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (Cfg::kRepOk && threadIdx.x < 128) tau_sh[threadIdx.x] = ~0ull;  // no unit yet
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();  // the merge may be scheduled; it waits for this grid's partials

  if (warp == 0) {
    // ------------------------- TMA producer -------------------------
    // The (unit, n-tile, k-block) sequence of this CTA.  W does not depend on
    // the kernel launched before this one (the row gather), so the first S
    // stages get their W slices before the grid-dependency wait; their A
    // slices (the gathered rows) follow it.
    if (lane == 0) {
      prefetch_tmap(&tmap_a);
      prefetch_tmap(&tmap_b);
      int u = blockIdx.x, m_tile = 0, n = 0, n_end = 0, kb = 0;
      bool valid = false;
      auto start_unit = [&]() {
        valid = false;
        for (; u < a.num_units; u += gridDim.x) {
          m_tile = u % a.m_tiles;
          n = (u / a.m_tiles) * a.tiles_per_split;
          n_end = min(n + a.tiles_per_split, a.n_tiles);
          if (n < n_end) {
            valid = true;
            return;
          }
        }
      };
      auto advance = [&]() {
        if (++kb == k_blocks) {
          kb = 0;
          if (++n == n_end) {
            u += gridDim.x;
            start_unit();
          }
        }
      };
      // the stage's W slice: one [256 x 64] box, or with W stored [H x V] four [64 x 64]
      // boxes (64 vocabulary columns x 64 hidden rows each)
      auto load_b = [&](int s, int kb_, int n_) {
        if constexpr (kHV) {
#pragma unroll
          for (int j = 0; j < kBN / 64; ++j)
            tma_load_2d(sB + s * kStageBytesB + j * kHvBlockBytes, &tmap_b, n_ * kBN + 64 * j, kb_ * kBK, &full[s]);
        } else {
          tma_load_2d(sB + s * kStageBytesB, &tmap_b, kb_ * kBK, n_ * kBN, &full[s]);
        }
      };
      start_unit();
      int pm[S], pk[S];
      int np = 0;
      uint32_t n_issued = 0;  // stage loads issued: load i went to stage i % S, phase (i / S) & 1
#pragma unroll
      for (int j = 0; j < S; ++j) {
        if (valid) {  // a fresh ring: the empty barriers need no wait yet
          pm[j] = m_tile;
          pk[j] = kb;
          mbar_arrive_expect_tx(&full[j], a.a_bytes + kStageBytesB);
          load_b(j, kb, n);
          advance();
          np = j + 1;
          ++n_issued;
        }
      }
      // During the grid-dependency wait: the next kWaitPrefetch W slices into L2, by the CTAs
      // of the first row tile only (the other row tiles read the same slices).
      {
        const int su = u, smt = m_tile, sn = n, sne = n_end, skb = kb;
        const bool sv = valid;
        for (int j = 0; j < kWaitPrefetch && valid; ++j) {
          if (m_tile == 0) {
            if constexpr (kHV) {
#pragma unroll
              for (int q = 0; q < kBN / 64; ++q) tma_prefetch_l2_2d(&tmap_b, n * kBN + 64 * q, kb * kBK);
            } else {
              tma_prefetch_l2_2d(&tmap_b, kb * kBK, n * kBN);
            }
          }
          advance();
        }
        u = su;
        m_tile = smt;
        n = sn;
        n_end = sne;
        kb = skb;
        valid = sv;
      }
      // the stage's A slice: one box, or with the column split one box per row copy
      auto load_a = [&](int s, int kb_, int m_tile_) {
        if (a.rep > 1) {
          for (int p = 0; p < a.rep; ++p)
            tma_load_2d(sA + s * Cfg::kStageA + p * a.rep_nq * 32 * 128, &tmap_a, kb_ * kBK, 0, &full[s]);
        } else {
          tma_load_2d(sA + s * Cfg::kStageA, &tmap_a, kb_ * kBK, m_tile_ * kBM, &full[s]);
        }
      };
      pdl_wait();  // the gathered rows are written by the preceding kernel
#pragma unroll
      for (int j = 0; j < S; ++j)
        if (j < np) load_a(j, pk[j], pm[j]);
      int s = np == S ? 0 : np;
      uint32_t ph = np == S ? 1u : 0u;
      while (valid) {
        if (!wait_or_abort(&empty[s], ph ^ 1u, abort_flag, a.dev_status, a.wait_ns)) break;
        mbar_arrive_expect_tx(&full[s], a.a_bytes + kStageBytesB);
        load_a(s, kb, m_tile);
        load_b(s, kb, n);
        advance();
        ++n_issued;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Every stage's last load lands before the CTA exits (after an abort some may
      // still be in flight; otherwise these waits return at once).  Full limit.
      for (uint32_t i = n_issued > static_cast<uint32_t>(S) ? n_issued - S : 0u; i < n_issued; ++i)
        mbar_wait(&full[i % S], (i / S) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------- MMA issuer -------------------------
    if (lane == 0) {
      uint32_t t = 0;
      int s = 0;
      uint32_t ph = 0;
      bool live = true;
      for (int u = blockIdx.x; u < a.num_units && live; u += gridDim.x) {
        const int split = u / a.m_tiles;
        const int n_begin = split * a.tiles_per_split;
        const int n_end = min(n_begin + a.tiles_per_split, a.n_tiles);
        for (int n = n_begin; n < n_end && live; ++n, ++t) {
          const uint32_t b = t & 1u, aph = (t >> 1) & 1u;
          if (!wait_or_abort(&acc_empty[b], aph ^ 1u, abort_flag, a.dev_status, a.wait_ns)) {
            live = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * kBN;
          for (int kb = 0; kb < k_blocks; ++kb) {
            if (!wait_or_abort(&full[s], ph, abort_flag, a.dev_status, a.wait_ns)) {
              live = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + s * Cfg::kStageA);
            const uint32_t b_addr = smem_u32(sB + s * kStageBytesB);
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
              const uint64_t ad = sw128_kmajor_desc(a_addr + kk * kUmmaK * 2);
              if constexpr (kHV) {  // W stored [H x V]: the slice is vocabulary-major
                const uint64_t bd = sw128_mnmajor_desc(b_addr + kk * kUmmaK * 128);
                umma_bf16(d_tmem, ad, bd, (kb > 0 || kk > 0) ? 1u : 0u, kIdescBmn);
              } else {
                const uint64_t bd = sw128_kmajor_desc(b_addr + kk * kUmmaK * 2);
                umma_bf16(d_tmem, ad, bd, (kb > 0 || kk > 0) ? 1u : 0u);
              }
            }
            umma_commit(&empty[s]);
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (live) umma_commit(&acc_full[b]);
        }
      }
      // Every MMA this thread issued has completed before the tensor memory is freed
      // (after an abort some may still run; otherwise the wait returns at once).
      umma_commit(mma_drain);
      mbar_wait(mma_drain, 0);
    }
  } else {
    // ------------------------- epilogue -------------------------
    const int q = warp & 3;  // TMEM lane quarter of this warp
    // column split (small batches): this warp's row copy and its first 64-column block
    const int n_rep = Cfg::kRepOk ? a.rep : 1;
    const int copy = n_rep > 1 ? q / a.rep_nq : 0;
    const int r_local = (n_rep > 1 ? q % a.rep_nq : q) * 32 + lane;  // row within the tile
    const float L = kLog2e;
    uint32_t t = 0, xu = 0;
    // With fewer than 128 rows (one row tile) the quarters beyond the last
    // row have nothing to read: their warps go straight to the final barrier
    // instead of polling the accumulator barriers (they are not counted there).
    bool live = q < a.epi_quarters;
    for (int u = blockIdx.x; u < a.num_units && live; u += gridDim.x) {
      const int m_tile = u % a.m_tiles, split = u / a.m_tiles;
      const int n_begin = split * a.tiles_per_split;
      const int n_end = min(n_begin + a.tiles_per_split, a.n_tiles);
      const int row = m_tile * kBM + r_local;
      const bool valid = row < a.rows;
      const bool warp_active = (m_tile * kBM + (r_local & ~31)) < a.rows;
      int k_row = 0, sel_id = -1;
      if (valid) {
        k_row = a.k_max;
        if (a.row_k) k_row = min(max(a.row_k[row], 0), a.k_max);
        if (a.sel) sel_id = a.sel[row];
      }
      float m = -INFINITY, ssum = 0.0f, sel_val = 0.0f;
      bool has_sel = false;
      // sampling: the row's best score z/T + g (greedy: z) over the allowed tokens so far
      float s_best = -INFINITY, s_z = -INFINITY, s_inv_t = 0.0f;
      int32_t s_id = -1;
      bool s_greedy = true;
      uint32_t s_off_lo = 0, s_off_hi = 0;
      if (kSamp != kSampNone && valid) {
        const float T = a.samp.temperature ? a.samp.temperature[row] : 1.0f;
        s_greedy = !(T > 0.0f);
        s_inv_t = s_greedy ? 0.0f : 1.0f / T;
        const uint64_t off = a.samp.offsets ? static_cast<uint64_t>(a.samp.offsets[row]) : static_cast<uint64_t>(row);
        s_off_lo = static_cast<uint32_t>(off);
        s_off_hi = static_cast<uint32_t>(off >> 32);
      }
      HeapState st;  // shared-memory heap (KCAP 128)
      st.tau = -INFINITY;
      st.cnt = 0;
      RegTopK<Cfg::kRegList ? KCAP : 1> rt;  // register list (KCAP <= 32)
      rt.reset();
      for (int n = n_begin; n < n_end; ++n, ++t) {
        const uint32_t b = t & 1u, aph = (t >> 1) & 1u;
        if (!wait_or_abort(&acc_full[b], aph, abort_flag, a.dev_status, a.wait_ns)) {
          live = false;
          break;
        }
        tc_fence_after();
        // The accumulator is handed back to the MMA as soon as this warp's last block of
        // the tile is in registers, so the next tile can start while that block is reduced.
        bool released = false;
        if (warp_active) {
          const int last_c = copy + ((kBN / kBlock - 1 - copy) / n_rep) * n_rep;
#pragma unroll 1
          for (int c = copy; c < kBN / kBlock; c += n_rep) {
            const int col0 = n * kBN + c * kBlock;
            if (col0 >= a.V) break;  // uniform across the warp
            float v[kBlock];
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * kBN + c * kBlock;
            __syncwarp();
            tmem_ld64(taddr, v);  // waits for the load (tcgen05.wait::ld)
            if (c == last_c) {
              tc_fence_before();
              mbar_arrive(&acc_empty[b]);
              released = true;
            }
            if (a.logit_scale != 1.0f) {  // head transform, applied before everything else reads the logits
#pragma unroll
              for (int j = 0; j < kBlock; ++j) v[j] *= a.logit_scale;
            }
            const int nvalid = a.V - col0;
            if (nvalid < kBlock) {
#pragma unroll
              for (int j = 0; j < kBlock; ++j)
                if (j >= nvalid) v[j] = -INFINITY;
            }
            const unsigned valid_mask = __ballot_sync(0xffffffffu, valid);  // whole warp converged here
            if (!valid) continue;
            if (kMaterialize) {
              float* dst = a.logits_out + static_cast<int64_t>(row) * a.V + col0;
              if ((a.V & 3) == 0 && nvalid >= kBlock) {
#pragma unroll
                for (int j = 0; j < kBlock; j += 4)
                  *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < kBlock; ++j)
                  if (j < nvalid) dst[j] = v[j];
              }
            }
            // block max and exp-sum as 8 and 4 independent chains (one warp runs this alone)
            float tm[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) tm[i] = v[i];
#pragma unroll
            for (int j = 8; j < kBlock; ++j) tm[j & 7] = fmaxf(tm[j & 7], v[j]);
            const float bm = fmaxf(fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3])),
                                   fmaxf(fmaxf(tm[4], tm[5]), fmaxf(tm[6], tm[7])));
            if (bm > m) {
              ssum *= ex2_approx((m - bm) * L);
              m = bm;
            }
            // exp(x - m) = 2^(x log2e - m log2e): one packed FFMA2 and one packed FADD2 per
            // pair of logits around the two ex2
            const float2 L2 = make_float2(L, L), nmL2 = make_float2(-m * L, -m * L);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int j = 0; j < kBlock; j += 2) {
              const float2 y = __ffma2_rn(make_float2(v[j], v[j + 1]), L2, nmL2);
              acc[(j >> 1) & 3] = __fadd2_rn(acc[(j >> 1) & 3], make_float2(ex2_approx(y.x), ex2_approx(y.y)));
            }
            const float2 a2 = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
            ssum += a2.x + a2.y;
            const int gcol0 = col0 + a.id_off;  // token id of the block's first logit
            const unsigned rel = static_cast<unsigned>(sel_id - gcol0);
            if (rel < static_cast<unsigned>(kBlock)) {
              float sv = 0.0f;
#pragma unroll
              for (int j = 0; j < kBlock; ++j) sv = (static_cast<unsigned>(j) == rel) ? v[j] : sv;
              sel_val = sv;
              has_sel = true;
            }
            if constexpr (kSamp != kSampNone) {
              // Gumbel-max over the block's allowed tokens; ids ascend, so ">" keeps the smaller id
              uint64_t allow = ~0ull;
              if (a.samp.mask) {
                const uint32_t* mrow = a.samp.mask + static_cast<int64_t>(row) * a.samp.mask_words;
                const int wd = col0 >> 5;
                allow = mrow[wd];
                if (wd + 1 < a.samp.mask_words) allow |= static_cast<uint64_t>(mrow[wd + 1]) << 32;
              }
              if (s_greedy) {
                if (bm > s_best) {
#pragma unroll
                  for (int j = 0; j < kBlock; ++j)
                    if (((allow >> j) & 1ull) && v[j] > s_best) {
                      s_best = v[j];
                      s_z = v[j];
                      s_id = col0 + j;
                    }
                }
              } else if (fmaf(bm, s_inv_t, kGumbelMax) > s_best) {  // else no token of the block can win
                const uint2 key = make_uint2(static_cast<uint32_t>(a.samp.seed), static_cast<uint32_t>(a.samp.seed >> 32));
                if constexpr (kSamp == kSampAll) {
#pragma unroll
                  for (int g4 = 0; g4 < kBlock / 4; ++g4) {
                    const uint4 w = philox4x32_10(
                        make_uint4(static_cast<uint32_t>(col0 >> 2) + g4, s_off_lo, s_off_hi, 0x53414D50u), key);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const int j = 4 * g4 + e;
                      const float sc = fmaf(v[j], s_inv_t, gumbel_of(ws[e]));
                      if (((allow >> j) & 1ull) && sc > s_best) {
                        s_best = sc;
                        s_z = v[j];
                        s_id = col0 + j;
                      }
                    }
                  }
                } else {
                  // pass 1: the words of every 4-token group; keep the allowed tokens whose word
                  // passes the candidate test for t = s_best - bm / T (the least noise that can win)
                  const uint32_t lim = noise_word_limit(s_best - bm * s_inv_t);
                  uint64_t cand = 0;
#pragma unroll
                  for (int g4 = 0; g4 < kBlock / 4; ++g4) {
                    const uint4 w = philox4x32_10(
                        make_uint4(static_cast<uint32_t>(col0 >> 2) + g4, s_off_lo, s_off_hi, 0x53414D50u), key);
                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                      cand |= static_cast<uint64_t>((0x800000u - (ws[e] >> 9)) < lim) << (4 * g4 + e);
                  }
                  cand &= allow;
                  if (cand) {
                    // pass 2, in id order: exact scores of the candidates (their group's words again;
                    // a logit is picked out of the registers by a select chain over the groups)
                    while (cand) {
                      const int g4 = (__ffsll(static_cast<long long>(cand)) - 1) >> 2;
                      const uint32_t gm = static_cast<uint32_t>(cand >> (4 * g4)) & 0xFu;
                      cand &= ~(0xFull << (4 * g4));
                      const uint4 w = philox4x32_10(
                          make_uint4(static_cast<uint32_t>(col0 >> 2) + g4, s_off_lo, s_off_hi, 0x53414D50u), key);
                      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                      for (int e = 0; e < 4; ++e) {
                        if ((gm >> e) & 1u) {
                          const int j = 4 * g4 + e;
                          float x = 0.0f;
#pragma unroll
                          for (int gg = 0; gg < kBlock / 4; ++gg) x = (gg == g4) ? v[4 * gg + e] : x;
                          const float sc = fmaf(x, s_inv_t, gumbel_of(ws[e]));
                          if (sc > s_best) {
                            s_best = sc;
                            s_z = x;
                            s_id = col0 + j;
                          }
                        }
                      }
                    }
                  }
                }
              }
            }
            if constexpr (Cfg::kRegList) {
              // Candidates: above this copy's own threshold, and not below any other copy's
              // (another copy's KCAP-th value bounds the row's KCAP-th value from below;
              // ">=" there keeps a tie that the smaller id may still win).
              float thr = rt.tau;
              if (Cfg::kRepOk && n_rep > 1) {
                float ts = -INFINITY;
                for (int p = 0; p < n_rep; ++p) {
                  if (p == copy) continue;
                  const uint64_t w = tau_sh[((q % a.rep_nq) + p * a.rep_nq) * 32 + lane];
                  if (static_cast<uint32_t>(w >> 32) == static_cast<uint32_t>(u))
                    ts = fmaxf(ts, __uint_as_float(static_cast<uint32_t>(w)));
                }
                thr = fmaxf(thr, float_below(ts));
              }
              // Stage the block for the lanes that have candidates; each lane then walks only its
              // own candidate mask, so the warp pays the largest per-lane count, not their union.
              const bool want = k_row > 0 && bm > thr;
              if (__any_sync(valid_mask, want)) {
                // staging: logit j of a lane at [j / 4][lane][j % 4] (16-byte stores, conflict-free)
                float* stg = reinterpret_cast<float*>(lists) + q * (kBlock * 32);
#pragma unroll
                for (int j = 0; j < kBlock; j += 4)
                  *reinterpret_cast<float4*>(stg + (j >> 2) * 128 + lane * 4) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                // candidate bits: the sign of thr - x is set exactly when x > thr (NaN and
                // -inf - -inf give a clear sign); funnel shifts collect one bit per logit,
                // the last logit first, so logit j lands on bit j
                const float2 t2 = make_float2(thr, thr), m1 = make_float2(-1.0f, -1.0f);
                uint32_t mlo = 0u, mhi = 0u;
#pragma unroll
                for (int j = kBlock - 2; j >= 0; j -= 2) {
                  const float2 d = __ffma2_rn(make_float2(v[j], v[j + 1]), m1, t2);
                  if (j >= 32) {
                    mhi = __funnelshift_l(__float_as_uint(d.y), mhi, 1);
                    mhi = __funnelshift_l(__float_as_uint(d.x), mhi, 1);
                  } else {
                    mlo = __funnelshift_l(__float_as_uint(d.y), mlo, 1);
                    mlo = __funnelshift_l(__float_as_uint(d.x), mlo, 1);
                  }
                }
                __syncwarp(valid_mask);
                uint64_t cm = want ? ((static_cast<uint64_t>(mhi) << 32) | mlo) : 0ull;
                while (cm) {
                  const int j = __ffsll(static_cast<long long>(cm)) - 1;
                  cm &= cm - 1;
                  const float x = stg[(j >> 2) * 128 + lane * 4 + (j & 3)];
                  if (x > rt.tau) rt.insert(x, gcol0 + j);
                }
                __syncwarp(valid_mask);
                if (Cfg::kRepOk && n_rep > 1 && want)
                  tau_sh[q * 32 + lane] = (static_cast<uint64_t>(static_cast<uint32_t>(u)) << 32) | __float_as_uint(rt.tau);
              }
            } else {
              if (k_row > 0 && bm > st.tau) {
#pragma unroll
                for (int j = 0; j < kBlock; ++j)
                  if (v[j] > st.tau) st = heap_push(lists, r_local, st, a.k_max, make_key(v[j], gcol0 + j));
              }
            }
          }
        }
        if (!released) {
          tc_fence_before();
          mbar_arrive(&acc_empty[b]);
        }
      }
      if (!live) break;
      // Column split: every copy's warp stages its row state and its sorted list (keys,
      // lane-interleaved) in its own staging region, now idle; the copy-0 warp of each lane
      // quarter folds the states into its own and merges the lists while writing them out.
      constexpr int KC = Cfg::kRegList ? KCAP : 1;
      const bool split_cols = Cfg::kRepOk && n_rep > 1;
      if (split_cols) {
        float* xs = reinterpret_cast<float*>(lists) + q * (kBlock * 32) + lane;
        uint64_t* xk = reinterpret_cast<uint64_t*>(lists) + q * (kBlock * 16) + 4 * 32 + lane;
#pragma unroll
        for (int j = 0; j < KC; ++j) xk[j * 32] = rt.key(j);
        if (copy > 0) {
          xs[0] = m;
          xs[32] = ssum;
          xs[64] = sel_val;
          xs[96] = has_sel ? 1.0f : 0.0f;
          xs[128] = s_best;
          xs[160] = __int_as_float(s_id);
          xs[192] = s_z;
          mbar_arrive(xchg_full);
          // the staging region is reused only after the leader has read it
          if (!wait_or_abort(xchg_empty, xu & 1u, abort_flag, a.dev_status, a.wait_ns)) break;
          ++xu;
          continue;
        }
        if (!wait_or_abort(xchg_full, xu & 1u, abort_flag, a.dev_status, a.wait_ns)) break;
        for (int p = 1; p < n_rep; ++p) {
          const float* ys = reinterpret_cast<const float*>(lists) + (q + p * a.rep_nq) * (kBlock * 32) + lane;
          const float mp = ys[0], sp = ys[32];
          if (mp > m) {
            ssum = ssum * ex2_approx((m - mp) * L) + sp;
            m = mp;
          } else if (mp != -INFINITY) {
            ssum += sp * ex2_approx((mp - m) * L);
          }
          if (ys[96] != 0.0f) {
            sel_val = ys[64];
            has_sel = true;
          }
          const float sb = ys[128];
          const int32_t sid = __float_as_int(ys[160]);
          if (sid >= 0 && (sb > s_best || (sb == s_best && (s_id < 0 || sid < s_id)))) {
            s_best = sb;
            s_id = sid;
            s_z = ys[192];
          }
        }
      }
      // f(j, key) for the row's best k_row keys, best first (key 0: fewer candidates)
      auto emit_keys = [&](auto&& f) {
        if constexpr (Cfg::kRegList) {
          if (split_cols) {
            // merge of the copies' sorted lists; keys are unique, so the best head is the one popped
            const uint64_t* xk = reinterpret_cast<const uint64_t*>(lists) + 4 * 32 + lane;
            const int w1 = (q + a.rep_nq) * (kBlock * 16), w2 = (q + 2 * a.rep_nq) * (kBlock * 16),
                      w3 = (q + 3 * a.rep_nq) * (kBlock * 16), w0 = q * (kBlock * 16);
            const bool four = n_rep > 2;
            int h0 = 0, h1 = 0, h2 = 0, h3 = 0;
            uint64_t k0 = xk[w0], k1 = xk[w1], k2 = four ? xk[w2] : 0ull, k3 = four ? xk[w3] : 0ull;
            // merged into registers first, written out after; each pop is branch-free (one
            // load from the popped list), so lanes that pop different lists do not diverge
            uint64_t res[KC];
#pragma unroll
            for (int j = 0; j < KC; ++j) {
              const uint64_t best = max(max(k0, k1), max(k2, k3));
              res[j] = best;
              if (j + 1 < KC) {
                const bool p0 = best == k0, p1 = !p0 && best == k1, p2 = !p0 && !p1 && best == k2;
                const int hp = (p0 ? h0 : p1 ? h1 : p2 ? h2 : h3) + 1;
                const int wp = p0 ? w0 : p1 ? w1 : p2 ? w2 : w3;
                const uint64_t nk = (hp < KC && best != 0ull) ? xk[wp + hp * 32] : 0ull;
                const bool p3 = !p0 && !p1 && !p2;
                k0 = p0 ? nk : k0;
                h0 = p0 ? hp : h0;
                k1 = p1 ? nk : k1;
                h1 = p1 ? hp : h1;
                k2 = p2 ? nk : k2;
                h2 = p2 ? hp : h2;
                k3 = p3 ? nk : k3;
                h3 = p3 ? hp : h3;
              }
            }
#pragma unroll
            for (int j = 0; j < KC; ++j)
              if (j < k_row) f(j, res[j]);
          } else {
#pragma unroll
            for (int j = 0; j < KC; ++j)
              if (j < k_row) f(j, rt.key(j));
          }
        } else {
          heap_sort_desc(lists, r_local, st.cnt);
          for (int j = 0; j < k_row; ++j) f(j, (j < st.cnt) ? lists[j * kBM + r_local] : 0ull);
        }
      };
      if (valid && a.final_out) {
        // the whole row went through this thread: lse = m + log(sum), logprob = logit - lse
        const float lse = (m == -INFINITY) ? -INFINITY : m + logf(ssum);
        a.out.lse[row] = lse;
        if (a.sel) {
          float sv = __int_as_float(0x7fc00000);  // NaN: no selected token / out of range
          if (sel_id >= 0 && sel_id < a.V)
            sv = sel_val - lse;
          else if (sel_id != -1)
            set_status(a.dev_status, LMH_DS_SEL_OUT_OF_RANGE);
          a.out.sel_logprob[row] = sv;
        }
        int32_t* ids = a.out.topk_ids + static_cast<int64_t>(row) * a.k_max;
        float* lps = a.out.topk_logprobs + static_cast<int64_t>(row) * a.k_max;
        auto put = [&](int j, uint64_t key) {  // key 0: fewer than k candidates
          ids[j] = key ? key_id(key) : -1;
          lps[j] = key ? key_value(key) - lse : -INFINITY;
        };
        emit_keys(put);
        for (int j = k_row; j < a.k_max; ++j) put(j, 0ull);
        if (kSamp != kSampNone) {
          a.samp.ids_out[row] = s_id;
          if (a.samp.lp_out) a.samp.lp_out[row] = s_id >= 0 ? s_z - lse : __int_as_float(0x7fc00000);
          if (s_id < 0) set_status(a.dev_status, LMH_DS_NO_ALLOWED_TOKEN);
        }
      } else if (valid) {
        const int64_t pidx = static_cast<int64_t>(row) * a.splits + split;
        a.parts.part_ms[pidx] = make_float2(m, ssum);
        unsigned long long* out = a.parts.part_keys + pidx * a.k_max;
        emit_keys([&](int j, uint64_t key) { out[j] = key; });
        if (has_sel) a.parts.sel_logit[row] = sel_val;
        if (kSamp != kSampNone) a.parts.part_samp[pidx] = make_float4(s_best, __int_as_float(s_id), s_z, 0.0f);
      }
      if (split_cols) {  // the copies' staging regions are free again
        mbar_arrive(xchg_empty);
        ++xu;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// per-mode entry points (instantiated in head_inst_*.cu)
// ---------------------------------------------------------------------------
template <int kSamp, bool kHV>
cudaError_t head_attr_mode() {
  cudaError_t e = cudaSuccess;
  auto set = [&](auto kernel, size_t smem) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  };
#define LMH_HEAD_ATTR(KC)                                                      \
  set(head_logprobs_kernel<KC, false, kSamp, false, kHV>, HeadCfg<KC>::kSmem); \
  set(head_logprobs_kernel<KC, true, kSamp, false, kHV>, HeadCfg<KC>::kSmem);
  LMH_HEAD_ATTR(1)
  LMH_HEAD_ATTR(5)
  LMH_HEAD_ATTR(8)
  LMH_HEAD_ATTR(16)
  LMH_HEAD_ATTR(20)
  LMH_HEAD_ATTR(32)
  LMH_HEAD_ATTR(128)
#undef LMH_HEAD_ATTR
  if constexpr (kSamp == kSampNone) {
#define LMH_HEAD_ATTR_DEEP(KC)                                                 \
  set(head_logprobs_kernel<KC, false, kSamp, true, kHV>, HeadCfg<KC, true>::kSmem); \
  set(head_logprobs_kernel<KC, true, kSamp, true, kHV>, HeadCfg<KC, true>::kSmem);
    LMH_HEAD_ATTR_DEEP(1)
    LMH_HEAD_ATTR_DEEP(5)
    LMH_HEAD_ATTR_DEEP(8)
    LMH_HEAD_ATTR_DEEP(16)
    LMH_HEAD_ATTR_DEEP(20)
    LMH_HEAD_ATTR_DEEP(32)
#undef LMH_HEAD_ATTR_DEEP
  }
  return e;
}

template <int kSamp, bool kHV>
cudaError_t launch_head_mode(int kcap, bool materialize, bool deep, dim3 grid, cudaStream_t stream, bool pdl,
                             const CUtensorMap& ta, const CUtensorMap& tb, const HeadArgs& a) {
  const dim3 block(kHeadThreads);
  if constexpr (kSamp == kSampNone) {
    if (deep) {
      switch (kcap) {
#define LMH_HEAD_CASE_DEEP(KC)                                                                                   \
  case KC:                                                                                                       \
    return materialize ? launch_kernel(head_logprobs_kernel<KC, true, kSamp, true, kHV>, grid, block,            \
                                       HeadCfg<KC, true>::kSmem, stream, pdl, ta, tb, a)                         \
                       : launch_kernel(head_logprobs_kernel<KC, false, kSamp, true, kHV>, grid, block,           \
                                       HeadCfg<KC, true>::kSmem, stream, pdl, ta, tb, a);
        LMH_HEAD_CASE_DEEP(1)
        LMH_HEAD_CASE_DEEP(5)
        LMH_HEAD_CASE_DEEP(8)
        LMH_HEAD_CASE_DEEP(16)
        LMH_HEAD_CASE_DEEP(20)
        LMH_HEAD_CASE_DEEP(32)
#undef LMH_HEAD_CASE_DEEP
        default:
          return cudaErrorInvalidValue;
      }
    }
  } else if (deep) {
    return cudaErrorInvalidValue;
  }
  switch (kcap) {
#define LMH_HEAD_CASE(KC)                                                                                      \
  case KC:                                                                                                     \
    return materialize ? launch_kernel(head_logprobs_kernel<KC, true, kSamp, false, kHV>, grid, block,          \
                                       HeadCfg<KC>::kSmem, stream, pdl, ta, tb, a)                             \
                       : launch_kernel(head_logprobs_kernel<KC, false, kSamp, false, kHV>, grid, block,         \
                                       HeadCfg<KC>::kSmem, stream, pdl, ta, tb, a);
    LMH_HEAD_CASE(1)
    LMH_HEAD_CASE(5)
    LMH_HEAD_CASE(8)
    LMH_HEAD_CASE(16)
    LMH_HEAD_CASE(20)
    LMH_HEAD_CASE(32)
    LMH_HEAD_CASE(128)
#undef LMH_HEAD_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

#define LMH_HEAD_MODE_DECL(EXT, MODE, HV)                                                                       \
  EXT template cudaError_t head_attr_mode<MODE, HV>();                                                          \
  EXT template cudaError_t launch_head_mode<MODE, HV>(int, bool, bool, dim3, cudaStream_t, bool,               \
                                                      const CUtensorMap&, const CUtensorMap&, const HeadArgs&);

}  // namespace lmh
