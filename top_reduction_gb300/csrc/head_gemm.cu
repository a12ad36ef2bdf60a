// head_gemm.cu -- selective head projection with a fused per-row reduction:
// the row gather (K2), the launch plan, the tensor maps and the launch of the
// tcgen05 head kernel (K3, head_kernel.cuh) in the mode the call needs.
//
// vllm-metal release v0.4.0.dev20260831, "Summary": gather the sampled rows
// and run the head on those alone.  MTPLX PR #532, "Change" and openinfer
// issue #719, "Suggested direction": per row one fp32 logsumexp, the selected
// token's logprob and the exact top-k, returned as an O(k+1) result; for
// finite k the [rows x vocab] logits are never written to memory.

#include <mutex>
#include <type_traits>

#include "head_kernel.cuh"

namespace lmh {

LMH_HEAD_MODE_DECL(extern, kSampNone, false)
LMH_HEAD_MODE_DECL(extern, kSampAll, false)
LMH_HEAD_MODE_DECL(extern, kSampFiltered, false)
LMH_HEAD_MODE_DECL(extern, kSampNone, true)
LMH_HEAD_MODE_DECL(extern, kSampAll, true)
LMH_HEAD_MODE_DECL(extern, kSampFiltered, true)

// ---------------------------------------------------------------------------
// row gather (K2): out[i, :] = hidden[row_idx[i], :]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ hidden, int64_t stride,
                                                          int num_tokens, const int32_t* __restrict__ row_idx,
                                                          int H, uint16_t* __restrict__ out, uint32_t* dev_status) {
  pdl_launch_dependents();  // the head kernel may start and stream W meanwhile
  pdl_wait();               // row_idx comes from the kernel launched just before
  const int i = blockIdx.x;
  const int src = row_idx ? row_idx[i] : i;
  const bool ok = src >= 0 && src < num_tokens;
  if (!ok && threadIdx.x == 0) set_status(dev_status, LMH_DS_ROW_IDX_OUT_OF_RANGE);
  uint16_t* dst = out + static_cast<int64_t>(i) * H;
  const uint16_t* s = hidden + static_cast<int64_t>(ok ? src : 0) * stride;
  const bool vec = ((stride & 7) == 0) && ((reinterpret_cast<uintptr_t>(hidden) & 15) == 0);
  if (vec) {
    const int nv = H / 8;
    for (int j = threadIdx.x; j < nv; j += blockDim.x)
      reinterpret_cast<uint4*>(dst)[j] = ok ? reinterpret_cast<const uint4*>(s)[j] : make_uint4(0, 0, 0, 0);
  } else {
    for (int j = threadIdx.x; j < H; j += blockDim.x) dst[j] = ok ? s[j] : static_cast<uint16_t>(0);
  }
}

cudaError_t launch_gather_rows(const void* hidden, int64_t hidden_stride, int num_tokens, const int32_t* row_idx,
                               int rows, int H, void* out, uint32_t* dev_status, cudaStream_t stream) {
  return launch_kernel(gather_rows_kernel, dim3(rows), dim3(256), 0, stream, true,
                       static_cast<const uint16_t*>(hidden), hidden_stride, num_tokens, row_idx, H,
                       static_cast<uint16_t*>(out), dev_status);
}

// ---------------------------------------------------------------------------
// host side: plan, tensor maps, launch
// ---------------------------------------------------------------------------

constexpr int kRepMaxH = 2048;  // hidden sizes from which lists of 16-20 need no column split

HeadPlan head_plan(int rows, int H, int V, int k_max, int num_sms) {
  HeadPlan p;
  p.m_tiles = (rows + kBM - 1) / kBM;
  p.n_tiles = (V + kBN - 1) / kBN;
  p.kcap = k_max <= 1    ? 1
           : k_max <= 5  ? 5
           : k_max <= 8  ? 8
           : k_max <= 16 ? 16
           : k_max <= 20 ? 20
           : k_max <= 32 ? 32
                         : 128;
  const int G = num_sms > 0 ? num_sms : 1;
  // Choose the vocabulary split that minimises the busiest CTA's tile count plus a cost
  // per unit.  A unit starts with empty candidate lists, so its first tile's reduction
  // takes about 23 us for 128 rows at K 20 (every logit of the first block enters the
  // list), against 4.5 us for later tiles.  With H below 2048 the MMA of two tiles
  // (5.4 us each at H 1024) cannot cover it and the unit start costs about two tiles;
  // with longer tiles only the flush and refill remain (a quarter of a tile).
  double best = 1e300;
  int best_s = 1;
  for (int s = 1; s <= p.n_tiles; ++s) {
    const int tps = (p.n_tiles + s - 1) / s;
    const int units = p.m_tiles * ((p.n_tiles + tps - 1) / tps);
    const int waves = (units + G - 1) / G;
    const double cost = static_cast<double>(waves) * (tps + (H < 2048 ? 2.0 : 0.25));
    if (cost < best - 1e-9) {
      best = cost;
      best_s = s;
    }
  }
  p.tiles_per_split = (p.n_tiles + best_s - 1) / best_s;
  p.splits = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  const int units = p.m_tiles * p.splits;
  p.grid = units < G ? units : G;
  return p;
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static cudaError_t get_encode(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  *fn = g_encode;
  return g_encode ? cudaSuccess : cudaErrorNotSupported;
}

// 2-D bf16 tensor map over a row-major [outer x inner] matrix with `pitch` elements per row.
static cudaError_t make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
                             uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  cudaError_t e = get_encode(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t head_setup() {
  cudaError_t e = head_attr_mode<kSampNone, false>();
  if (e == cudaSuccess) e = head_attr_mode<kSampAll, false>();
  if (e == cudaSuccess) e = head_attr_mode<kSampFiltered, false>();
  if (e == cudaSuccess) e = head_attr_mode<kSampNone, true>();
  if (e == cudaSuccess) e = head_attr_mode<kSampAll, true>();
  if (e == cudaSuccess) e = head_attr_mode<kSampFiltered, true>();
  return e;
}

cudaError_t launch_head(const void* A, int64_t a_stride, int rows, int H, const void* W, int V, const HeadPlan& plan,
                        const int32_t* sel, const int32_t* row_k, int k_max, Partials parts, float* logits_out,
                        uint32_t* dev_status, cudaStream_t stream, bool pdl, const RowOutputs* final_out,
                        float logit_scale, const SampleArgs* samp, bool w_hv, int id_off) {
  if (final_out && plan.splits != 1) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  // With fewer than 128 rows (one row tile) the A box covers only the real
  // rows (rounded up to 8); the stage's other rows keep stale data that only
  // reaches accumulator rows the epilogue never reads.
  const uint32_t a_box = rows < kBM ? static_cast<uint32_t>((rows + 7) / 8 * 8) : static_cast<uint32_t>(kBM);
  cudaError_t e = make_tmap(&ta, A, static_cast<uint64_t>(H), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(a_stride), kBK, a_box);
  if (e != cudaSuccess) return e;
  // W [V x H]: [256 x 64] boxes along H; W [H x V]: [64 x 64] boxes, vocabulary innermost
  e = w_hv ? make_tmap(&tb, W, static_cast<uint64_t>(V), static_cast<uint64_t>(H), static_cast<uint64_t>(V), 64, kBK)
           : make_tmap(&tb, W, static_cast<uint64_t>(H), static_cast<uint64_t>(V), static_cast<uint64_t>(H), kBK, kBN);
  if (e != cudaSuccess) return e;
  HeadArgs a;
  // Column split for batches of at most 64 rows with a heavy epilogue: sampling, or
  // lists of 16 or 20 entries on short tiles (H below kRepMaxH: the tile's W streams in
  // less time than one warp needs for the lists of its early blocks); longer lists do
  // not fit the exchange.  4 row copies of one lane quarter, or 2 of two.  Otherwise
  // one warp per lane quarter keeps up, and batches of at most 32 rows take the deep
  // layout (a deeper ring of W stages, HeadCfg<KCAP, true>), which pays more on an
  // HBM-bound head.
  a.rep = 1;
  a.rep_nq = 4;
  static_assert(HeadCfg<20>::kRepOk && !HeadCfg<32>::kRepOk, "column split: list capacities up to 20");
  const bool sampling = samp && samp->enabled;
  const bool rep_ok = plan.kcap <= 20 && (sampling || (plan.kcap >= 16 && H < kRepMaxH));
  if (rows >= 1 && rows <= 64 && rep_ok) {
    a.rep_nq = (rows + 31) / 32;
    a.rep = 4 / a.rep_nq;
  }
  const bool deep = !sampling && a.rep == 1 && rows <= 32 && plan.kcap <= 32;
  a.a_bytes = static_cast<uint32_t>(a.rep) * a_box * kBK * 2;
  a.rows = rows;
  a.H = H;
  a.V = V;
  a.k_max = k_max;
  a.m_tiles = plan.m_tiles;
  a.n_tiles = plan.n_tiles;
  a.splits = plan.splits;
  a.tiles_per_split = plan.tiles_per_split;
  a.num_units = plan.m_tiles * plan.splits;
  a.sel = sel;
  a.row_k = row_k;
  a.parts = parts;
  a.logits_out = logits_out;
  a.dev_status = dev_status;
  a.epi_quarters = a.rep > 1 ? 4 : (rows < kBM ? (rows + 31) / 32 : 4);
  a.logit_scale = logit_scale;
  a.samp = samp ? *samp : SampleArgs{};
  a.final_out = final_out ? 1 : 0;
  a.out = final_out ? *final_out : RowOutputs{nullptr, nullptr, nullptr, nullptr};
  a.wait_ns = wait_limit_ns();
  a.id_off = id_off;
  const dim3 grid(plan.grid);
  const bool mat = logits_out != nullptr;
  // the kernels for each weight layout: [V x H] (kHV false) or [H x V] (kHV true)
  auto launch = [&](auto mode, bool deep_) {
    constexpr int M = decltype(mode)::value;
    return w_hv ? launch_head_mode<M, true>(plan.kcap, mat, deep_, grid, stream, pdl, ta, tb, a)
                : launch_head_mode<M, false>(plan.kcap, mat, deep_, grid, stream, pdl, ta, tb, a);
  };
  if (!a.samp.enabled) return launch(std::integral_constant<int, kSampNone>{}, deep);
  // Sampling: the candidate filter pays off when a warp's rows see long vocabulary
  // ranges (its test tightens as the row's best score grows) or when few lanes hold
  // rows (a block's second pass runs for the lanes that have candidates); otherwise
  // every token is scored.  Both draw the same token.  Measured on GB300: 8 lanes x 4
  // blocks and 32 lanes x 184 blocks per unit favour the filter, 32 lanes x 4 and x 24
  // blocks favour scoring every token.
  const int lanes = plan.m_tiles == 1 ? (rows < 32 ? rows : 32) : 32;
  const int blocks_per_unit = plan.tiles_per_split * (kBN / 64) / a.rep;
  if (lanes <= 16 || blocks_per_unit >= 64)
    return launch(std::integral_constant<int, kSampFiltered>{}, false);
  return launch(std::integral_constant<int, kSampAll>{}, false);
}

}  // namespace lmh
