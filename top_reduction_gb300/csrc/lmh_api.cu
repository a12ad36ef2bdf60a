// lmh_api.cu -- the C ABI of liblmh: argument checks, workspace layout,
// one-time device set-up, kernel launches and the kernel trace.
//
// Nothing here computes results: every step of the path runs in the kernels
// of select_rows.cu, head_gemm.cu, logits_reduce.cu and merge_partials.cu.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "lmh.h"
#include "lmh_internal.h"

namespace lmh {

// ---------------------------------------------------------------------------
// per-device set-up
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
static std::mutex g_setup_mu;
static bool g_setup_done[kMaxDevices];
static int g_num_sms[kMaxDevices];

static cudaError_t device_setup(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_setup_done[dev]) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = logits_reduce_setup();
    if (e == cudaSuccess) e = merge_setup();
    if (e == cudaSuccess) e = head_setup();
    if (e != cudaSuccess) return e;
    g_num_sms[dev] = sms;
    g_setup_done[dev] = true;
  }
  *num_sms = g_num_sms[dev];
  return cudaSuccess;
}

static inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// limit of the kernels' bounded waits (read at every launch)
static std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

size_t partials_bytes(int rows, int splits, int k_max) {
  const size_t rs = static_cast<size_t>(rows) * static_cast<size_t>(splits);
  return align256(rs * 8) + align256(rs * static_cast<size_t>(k_max) * 8) + align256(static_cast<size_t>(rows) * 4) +
         align256(rs * 16);
}

Partials carve_partials(void* base, int rows, int splits, int k_max) {
  char* p = static_cast<char*>(base);
  const size_t rs = static_cast<size_t>(rows) * static_cast<size_t>(splits);
  Partials out;
  out.part_ms = reinterpret_cast<float2*>(p);
  p += align256(rs * 8);
  out.part_keys = reinterpret_cast<unsigned long long*>(p);
  p += align256(rs * static_cast<size_t>(k_max) * 8);
  out.sel_logit = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(rows) * 4);
  out.part_samp = reinterpret_cast<float4*>(p);
  out.bmax = nullptr;
  out.ticket = nullptr;
  return out;
}

// ---------------------------------------------------------------------------
// kernel trace
// ---------------------------------------------------------------------------
static const char* const kTraceNames[kTraceCount] = {"select_rows",    "gather_rows",   "head_logprobs",
                                                     "logits_reduce",  "merge_partials", "logits_select",
                                                     "full_logprobs"};

struct TraceRecord {
  int kernel;
  cudaEvent_t start, stop;
};

static std::mutex g_trace_mu;
static volatile bool g_trace_on = false;
static std::vector<TraceRecord> g_trace_pending;
static std::vector<cudaEvent_t> g_trace_pool;
static int64_t g_trace_launches[kTraceCount];
static double g_trace_ms[kTraceCount];
static thread_local cudaEvent_t t_open[kTraceCount];

static cudaEvent_t trace_take_event() {
  {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (!g_trace_pool.empty()) {
      cudaEvent_t e = g_trace_pool.back();
      g_trace_pool.pop_back();
      return e;
    }
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void trace_begin(TraceKernel k, cudaStream_t s) {
  if (!g_trace_on) return;
  cudaEvent_t e = trace_take_event();
  if (e && cudaEventRecord(e, s) == cudaSuccess) t_open[k] = e;
}

void trace_end(TraceKernel k, cudaStream_t s) {
  cudaEvent_t start = t_open[k];
  if (!start) return;
  t_open[k] = nullptr;
  cudaEvent_t stop = trace_take_event();
  if (!stop || cudaEventRecord(stop, s) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(g_trace_mu);
  g_trace_pending.push_back({static_cast<int>(k), start, stop});
}

static lmh_status trace_drain() {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  lmh_status st = LMH_OK;
  for (const TraceRecord& r : g_trace_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
      st = LMH_ERR_CUDA;
    g_trace_launches[r.kernel] += 1;
    g_trace_ms[r.kernel] += ms;
    g_trace_pool.push_back(r.start);
    g_trace_pool.push_back(r.stop);
  }
  g_trace_pending.clear();
  return st;
}

// RAII bracket for one traced launch
struct Traced {
  TraceKernel k;
  cudaStream_t s;
  Traced(TraceKernel k_, cudaStream_t s_) : k(k_), s(s_) { trace_begin(k, s); }
  ~Traced() { trace_end(k, s); }
};

static lmh_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LMH_OK : LMH_ERR_CUDA; }

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspace of lmh_probe_selective: the projection's own workspace (k_max 0),
// then the materialized logits f32 [rows x V] and an lse [rows].
static size_t probe_project_bytes(int rows, int hidden, int vocab, int sms) {
  const HeadPlan p = head_plan(rows, hidden, vocab, 0, sms);
  return align256(static_cast<size_t>(rows) * static_cast<size_t>(hidden) * 2) + partials_bytes(rows, p.splits, 0);
}
static size_t probe_bytes(int rows, int hidden, int vocab, int sms) {
  if (hidden <= 0) return 0;
  return probe_project_bytes(rows, hidden, vocab, sms) +
         align256(static_cast<size_t>(rows) * static_cast<size_t>(vocab) * 4) + align256(static_cast<size_t>(rows) * 4);
}

}  // namespace lmh

using namespace lmh;

extern "C" {

int32_t lmh_version(void) { return LMH_VERSION; }

const char* lmh_status_string(lmh_status s) {
  switch (s) {
    case LMH_OK: return "LMH_OK";
    case LMH_ERR_INVALID_ARG: return "LMH_ERR_INVALID_ARG";
    case LMH_ERR_UNSUPPORTED: return "LMH_ERR_UNSUPPORTED";
    case LMH_ERR_WORKSPACE_TOO_SMALL: return "LMH_ERR_WORKSPACE_TOO_SMALL";
    case LMH_ERR_CUDA: return "LMH_ERR_CUDA";
    case LMH_ERR_TIMEOUT: return "LMH_ERR_TIMEOUT";
  }
  return "LMH_ERR_UNKNOWN";
}

lmh_status lmh_select_rows(const int32_t* cu_seqlens, int32_t num_seqs, int32_t num_decode,
                           const uint8_t* all_rows_mask, int32_t max_out_rows, int32_t* row_idx,
                           int32_t* logits_cu_seqlens, uint32_t* dev_status, cudaStream_t stream) {
  if (!cu_seqlens || !logits_cu_seqlens || num_seqs < 0 || num_decode < 0 || num_decode > num_seqs ||
      max_out_rows < 0 || (max_out_rows > 0 && !row_idx))
    return LMH_ERR_INVALID_ARG;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return LMH_ERR_CUDA;
  Traced tr(kTraceSelect, stream);
  return from_cuda(launch_select_rows(cu_seqlens, num_seqs, num_decode, all_rows_mask, max_out_rows, row_idx,
                                      logits_cu_seqlens, dev_status, stream));
}

int32_t lmh_count_selected_rows(const int32_t* cu, int32_t num_seqs, int32_t num_decode, const uint8_t* mask) {
  if (!cu || num_seqs < 0 || num_decode < 0 || num_decode > num_seqs) return -1;
  if (num_seqs > 0 && cu[0] != 0) return -1;
  int64_t n = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t lo = cu[s], hi = cu[s + 1];
    if (hi < lo) return -1;
    if (s < num_decode || (mask && mask[s]))
      n += hi - lo;
    else if (hi == lo)
      return -1;
    else
      n += 1;
  }
  return n > INT32_MAX ? -1 : static_cast<int32_t>(n);
}

size_t lmh_workspace_bytes(int32_t rows, int32_t hidden, int32_t vocab, int32_t k_max, lmh_path path) {
  if (k_max == LMH_K_FULL) k_max = 0;  // the full-vocabulary output needs the K 0 workspace
  if (rows < 0 || vocab <= 0 || k_max < 0 || k_max > LMH_K_MAX || k_max > vocab) return 0;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return 0;
  if (rows == 0) return 256;
  if (path == LMH_PATH_PROJECT) {
    if (hidden <= 0) return 0;
    const HeadPlan p = head_plan(rows, hidden, vocab, k_max, sms);
    return align256(static_cast<size_t>(rows) * static_cast<size_t>(hidden) * 2) +
           partials_bytes(rows, p.splits, k_max);
  }
  if (path == LMH_PATH_FROM_LOGITS) {
    const VocabSplit vs = logits_reduce_split(rows, vocab, k_max, sms);
    return stream_partials_bytes(rows, vs);
  }
  if (path == LMH_PATH_PROBE) return probe_bytes(rows, hidden, vocab, sms);
  return 0;
}

}  // extern "C"

// The projection with a head transform (logit_scale 1: none).
static lmh_status project_impl(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                               const int32_t* row_idx, int32_t rows, int32_t H, const void* W,
                               lmh_w_layout w_layout, int32_t V, const int32_t* sel_ids, const int32_t* row_k,
                               int32_t k_req, float* lse, float* sel_logprob, int32_t* topk_ids,
                               float* topk_logprobs, float* logits_out, void* workspace, size_t workspace_bytes,
                               uint32_t* dev_status, float logit_scale, cudaStream_t stream,
                               const SampleArgs* samp = nullptr) {
  if (rows < 0 || H <= 0 || V <= 0 || num_tokens < 0) return LMH_ERR_INVALID_ARG;
  if (k_req < LMH_K_FULL || k_req > LMH_K_MAX) return LMH_ERR_UNSUPPORTED;
  if (k_req > V) return LMH_ERR_INVALID_ARG;
  // Full-vocabulary output: the reduction runs with K 0 (lse, selected token)
  // and a pass writes z - lse; the fp32 logits are materialized in the output.
  const bool full = k_req == LMH_K_FULL;
  const int32_t k_max = full ? 0 : k_req;
  if (full && (!topk_logprobs || !aligned(topk_logprobs, 16))) return LMH_ERR_INVALID_ARG;
  float* z_out = (full && !logits_out) ? topk_logprobs : logits_out;
  if (w_layout != LMH_W_VH && w_layout != LMH_W_HV) return LMH_ERR_INVALID_ARG;
  if (!hidden || !W || !lse || (sel_ids && !sel_logprob) || (k_max > 0 && (!topk_ids || !topk_logprobs)))
    return LMH_ERR_INVALID_ARG;
  if (hidden_row_stride < H) return LMH_ERR_INVALID_ARG;
  if (!row_idx && rows > num_tokens) return LMH_ERR_INVALID_ARG;
  // W [H x V] rows are V elements: the tensor map wants them a multiple of 16 bytes
  if (w_layout == LMH_W_HV && (V % 8) != 0) return LMH_ERR_UNSUPPORTED;
  if ((H % 8) != 0 || !aligned(hidden, 16) || !aligned(W, 16) || (logits_out && !aligned(logits_out, 16)))
    return LMH_ERR_UNSUPPORTED;
  if (rows == 0) return LMH_OK;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return LMH_ERR_CUDA;
  const HeadPlan plan = head_plan(rows, H, V, k_max, sms);
  const size_t gather_bytes = align256(static_cast<size_t>(rows) * static_cast<size_t>(H) * 2);
  const size_t need = gather_bytes + partials_bytes(rows, plan.splits, k_max);
  if (!workspace || !aligned(workspace, 256)) return LMH_ERR_INVALID_ARG;
  if (workspace_bytes < need) return LMH_ERR_WORKSPACE_TOO_SMALL;

  char* ws = static_cast<char*>(workspace);
  const Partials parts = carve_partials(ws + gather_bytes, rows, plan.splits, k_max);
  const bool gather = row_idx != nullptr || (hidden_row_stride % 8) != 0;
  const void* A = hidden;
  int64_t a_stride = hidden_row_stride;
  cudaError_t e = cudaSuccess;
  if (gather) {
    Traced tr(kTraceGather, stream);
    e = launch_gather_rows(hidden, hidden_row_stride, num_tokens, row_idx, rows, H, ws, dev_status, stream);
    A = ws;
    a_stride = H;
  }
  // One vocabulary split: the head kernel finishes every row itself.  The head is always
  // launched with programmatic dependent launch: it streams its first W slices while the
  // kernel before it (the row gather, or the previous call's merge) ends.
  const RowOutputs outs{lse, sel_logprob, topk_ids, topk_logprobs};
  const bool one_split = plan.splits == 1;
  if (e == cudaSuccess) {
    Traced tr(kTraceHead, stream);
    e = launch_head(A, a_stride, rows, H, W, V, plan, sel_ids, row_k, k_max, parts, z_out, dev_status, stream,
                    /*pdl=*/true, one_split ? &outs : nullptr, logit_scale, samp, w_layout == LMH_W_HV);
  }
  if (e == cudaSuccess && !one_split) {
    Traced tr(kTraceMerge, stream);
    e = launch_merge(rows, plan.splits, V, k_max, parts, sel_ids, row_k, lse, sel_logprob, topk_ids, topk_logprobs,
                     dev_status, stream, /*pdl=*/true, samp, sms);
  }
  if (e == cudaSuccess && full)
    e = launch_full_logprobs(z_out, LMH_F32, V, rows, V, lse, topk_logprobs, stream);
  return from_cuda(e);
}

extern "C" {

lmh_status lmh_project_logprobs(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                const int32_t* row_idx, int32_t rows, int32_t H, const void* W,
                                lmh_w_layout w_layout, int32_t V, const int32_t* sel_ids, const int32_t* row_k,
                                int32_t k_max, float* lse, float* sel_logprob, int32_t* topk_ids,
                                float* topk_logprobs, float* logits_out, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_status, cudaStream_t stream) {
  return project_impl(hidden, hidden_row_stride, num_tokens, row_idx, rows, H, W, w_layout, V, sel_ids, row_k, k_max,
                      lse, sel_logprob, topk_ids, topk_logprobs, logits_out, workspace, workspace_bytes, dev_status,
                      1.0f, stream);
}

static bool valid_scale(float s) { return std::isfinite(s) && s > 0.0f; }

lmh_status lmh_project_logprobs_scaled(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                       const int32_t* row_idx, int32_t rows, int32_t H, const void* W,
                                       lmh_w_layout w_layout, int32_t V, const int32_t* sel_ids,
                                       const int32_t* row_k, int32_t k_max, float* lse, float* sel_logprob,
                                       int32_t* topk_ids, float* topk_logprobs, float* logits_out,
                                       void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                       float logit_scale, cudaStream_t stream) {
  if (!valid_scale(logit_scale)) return LMH_ERR_INVALID_ARG;
  return project_impl(hidden, hidden_row_stride, num_tokens, row_idx, rows, H, W, w_layout, V, sel_ids, row_k, k_max,
                      lse, sel_logprob, topk_ids, topk_logprobs, logits_out, workspace, workspace_bytes, dev_status,
                      logit_scale, stream);
}

lmh_status lmh_logprobs_from_logits(const void* logits, lmh_dtype dtype, int32_t rows, int32_t V, int64_t row_stride,
                                    const int32_t* sel_ids, const int32_t* row_k, int32_t k_max, float* lse,
                                    float* sel_logprob, int32_t* topk_ids, float* topk_logprobs, void* workspace,
                                    size_t workspace_bytes, uint32_t* dev_status, cudaStream_t stream) {
  if (rows < 0 || V <= 0 || row_stride < V) return LMH_ERR_INVALID_ARG;
  if (dtype != LMH_BF16 && dtype != LMH_F16 && dtype != LMH_F32) return LMH_ERR_INVALID_ARG;
  if (k_max < LMH_K_FULL || k_max > LMH_K_MAX) return LMH_ERR_UNSUPPORTED;
  if (k_max > V) return LMH_ERR_INVALID_ARG;
  if (!logits || !lse || (sel_ids && !sel_logprob) || (k_max > 0 && (!topk_ids || !topk_logprobs)))
    return LMH_ERR_INVALID_ARG;
  if (k_max == LMH_K_FULL && (!topk_logprobs || !aligned(topk_logprobs, 16))) return LMH_ERR_INVALID_ARG;
  const int64_t elem = dtype == LMH_F32 ? 4 : 2;
  if (!aligned(logits, static_cast<size_t>(elem))) return LMH_ERR_UNSUPPORTED;
  if (rows == 0) return LMH_OK;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return LMH_ERR_CUDA;
  const VocabSplit vs = logits_reduce_split(rows, V, k_max, sms);
  if (static_cast<int64_t>(rows) * vs.splits > INT32_MAX) return LMH_ERR_UNSUPPORTED;
  const size_t need = stream_partials_bytes(rows, vs);
  if (!workspace || !aligned(workspace, 256)) return LMH_ERR_INVALID_ARG;
  if (workspace_bytes < need) return LMH_ERR_WORKSPACE_TOO_SMALL;
  const Partials parts = carve_stream_partials(workspace, rows, vs);
  const cudaError_t e = launch_logits_reduce(logits, dtype, row_stride, rows, V, vs, sel_ids, row_k, k_max, parts,
                                             lse, sel_logprob, topk_ids, topk_logprobs, dev_status, stream);
  return from_cuda(e);
}

lmh_status lmh_project_logprobs_sample(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                       const int32_t* row_idx, int32_t rows, int32_t H, const void* W,
                                       lmh_w_layout w_layout, int32_t V, const int32_t* sel_ids,
                                       const int32_t* row_k, int32_t k_max, float* lse, float* sel_logprob,
                                       int32_t* topk_ids, float* topk_logprobs, float* logits_out,
                                       void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                       float logit_scale, const lmh_sampling* sampling, cudaStream_t stream) {
  if (!sampling || !sampling->sampled_ids || !valid_scale(logit_scale) || V <= 0) return LMH_ERR_INVALID_ARG;
  if (sampling->allowed_mask && sampling->mask_words < (V + 31) / 32) return LMH_ERR_INVALID_ARG;
  SampleArgs sa{};
  sa.enabled = 1;
  sa.temperature = sampling->temperature;
  sa.mask = sampling->allowed_mask;
  sa.mask_words = sampling->mask_words;
  sa.seed = sampling->seed;
  sa.offsets = sampling->offsets;
  sa.ids_out = sampling->sampled_ids;
  sa.lp_out = sampling->sampled_logprob;
  return project_impl(hidden, hidden_row_stride, num_tokens, row_idx, rows, H, W, w_layout, V, sel_ids, row_k, k_max,
                      lse, sel_logprob, topk_ids, topk_logprobs, logits_out, workspace, workspace_bytes, dev_status,
                      logit_scale, stream, &sa);
}

lmh_status lmh_probe_selective(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                               const int32_t* row_idx, int32_t rows, int32_t H, const void* W, int32_t V,
                               float logit_scale, const float* ref_logits, float tolerance, uint32_t* mismatches,
                               void* workspace, size_t workspace_bytes, uint32_t* dev_status, cudaStream_t stream) {
  if (!ref_logits || !mismatches || !(tolerance >= 0.0f) || !valid_scale(logit_scale)) return LMH_ERR_INVALID_ARG;
  if (rows < 0 || H <= 0 || V <= 0) return LMH_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return LMH_ERR_INVALID_ARG;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return LMH_ERR_CUDA;
  if (workspace_bytes < probe_bytes(rows, H, V, sms)) return LMH_ERR_WORKSPACE_TOO_SMALL;
  if (rows == 0) return from_cuda(cudaMemsetAsync(mismatches, 0, sizeof(uint32_t), stream));
  char* ws = static_cast<char*>(workspace);
  const size_t proj = probe_project_bytes(rows, H, V, sms);
  float* ours = reinterpret_cast<float*>(ws + proj);
  float* lse = reinterpret_cast<float*>(ws + proj + align256(static_cast<size_t>(rows) * static_cast<size_t>(V) * 4));
  const lmh_status st = project_impl(hidden, hidden_row_stride, num_tokens, row_idx, rows, H, W, LMH_W_VH, V, nullptr,
                                     nullptr, 0, lse, nullptr, nullptr, nullptr, ours, workspace, proj, dev_status,
                                     logit_scale, stream);
  if (st != LMH_OK) return st;
  return from_cuda(launch_probe_compare(ours, ref_logits, static_cast<int64_t>(rows) * V, tolerance, mismatches, sms,
                                        stream));
}

size_t lmh_record_bytes(int32_t k_max) {
  if (k_max < 0 || k_max > LMH_K_MAX) return 0;
  return record_bytes(k_max);
}

// One rank's share of a vocabulary-parallel head: the gather, the head over the
// share's rows of W (token ids offset by v_begin) and the merge of its vocabulary
// ranges into one record per row.
lmh_status lmh_project_partials(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                const int32_t* row_idx, int32_t rows, int32_t H, const void* W_share,
                                lmh_w_layout w_layout, int32_t v_begin, int32_t v_count, int32_t V,
                                const int32_t* sel_ids, const int32_t* row_k, int32_t k_max, void* records,
                                void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                cudaStream_t stream) {
  if (rows < 0 || H <= 0 || V <= 0 || num_tokens < 0 || v_begin < 0 || v_count <= 0 ||
      static_cast<int64_t>(v_begin) + v_count > V)
    return LMH_ERR_INVALID_ARG;
  if (k_max < 0 || k_max > LMH_K_MAX) return LMH_ERR_UNSUPPORTED;
  if (k_max > v_count) return LMH_ERR_INVALID_ARG;
  if (w_layout != LMH_W_VH) return LMH_ERR_UNSUPPORTED;
  if (!hidden || !W_share || !records || hidden_row_stride < H || (!row_idx && rows > num_tokens))
    return LMH_ERR_INVALID_ARG;
  if ((H % 8) != 0 || !aligned(hidden, 16) || !aligned(W_share, 16) || !aligned(records, 8))
    return LMH_ERR_UNSUPPORTED;
  if (rows == 0) return LMH_OK;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return LMH_ERR_CUDA;
  const HeadPlan plan = head_plan(rows, H, v_count, k_max, sms);
  const size_t gather_bytes = align256(static_cast<size_t>(rows) * static_cast<size_t>(H) * 2);
  const size_t need = gather_bytes + partials_bytes(rows, plan.splits, k_max);
  if (!workspace || !aligned(workspace, 256)) return LMH_ERR_INVALID_ARG;
  if (workspace_bytes < need) return LMH_ERR_WORKSPACE_TOO_SMALL;
  char* ws = static_cast<char*>(workspace);
  const Partials parts = carve_partials(ws + gather_bytes, rows, plan.splits, k_max);
  const bool gather = row_idx != nullptr || (hidden_row_stride % 8) != 0;
  const void* A = hidden;
  int64_t a_stride = hidden_row_stride;
  cudaError_t e = cudaSuccess;
  if (gather) {
    Traced tr(kTraceGather, stream);
    e = launch_gather_rows(hidden, hidden_row_stride, num_tokens, row_idx, rows, H, ws, dev_status, stream);
    A = ws;
    a_stride = H;
  }
  if (e == cudaSuccess) {
    Traced tr(kTraceHead, stream);
    e = launch_head(A, a_stride, rows, H, W_share, v_count, plan, sel_ids, row_k, k_max, parts, nullptr, dev_status,
                    stream, /*pdl=*/true, nullptr, 1.0f, nullptr, false, v_begin);
  }
  if (e == cudaSuccess) {
    const RecordOut rec{static_cast<unsigned char*>(records), v_begin, v_count};
    Traced tr(kTraceMerge, stream);
    e = launch_merge(rows, plan.splits, V, k_max, parts, sel_ids, row_k, nullptr, nullptr, nullptr, nullptr,
                     dev_status, stream, /*pdl=*/true, nullptr, sms, &rec);
  }
  return from_cuda(e);
}

size_t lmh_merge_workspace_bytes(int32_t rows, int32_t num_parts, int32_t k_max) {
  if (rows < 0 || num_parts <= 0 || k_max < 0 || k_max > LMH_K_MAX) return 0;
  if (rows == 0) return 256;
  return partials_bytes(rows, num_parts, k_max);
}

lmh_status lmh_merge_records(const void* records, int32_t num_parts, int32_t rows, int32_t V,
                             const int32_t* sel_ids, const int32_t* row_k, int32_t k_max, float* lse,
                             float* sel_logprob, int32_t* topk_ids, float* topk_logprobs, void* workspace,
                             size_t workspace_bytes, uint32_t* dev_status, cudaStream_t stream) {
  if (rows < 0 || num_parts <= 0 || V <= 0) return LMH_ERR_INVALID_ARG;
  if (k_max < 0 || k_max > LMH_K_MAX) return LMH_ERR_UNSUPPORTED;
  if (k_max > V) return LMH_ERR_INVALID_ARG;
  if (!records || !lse || (sel_ids && !sel_logprob) || (k_max > 0 && (!topk_ids || !topk_logprobs)))
    return LMH_ERR_INVALID_ARG;
  if (!aligned(records, 8)) return LMH_ERR_UNSUPPORTED;
  if (rows == 0) return LMH_OK;
  int sms = 0;
  if (device_setup(&sms) != cudaSuccess) return LMH_ERR_CUDA;
  if (!workspace || !aligned(workspace, 256)) return LMH_ERR_INVALID_ARG;
  if (workspace_bytes < partials_bytes(rows, num_parts, k_max)) return LMH_ERR_WORKSPACE_TOO_SMALL;
  const Partials parts = carve_partials(workspace, rows, num_parts, k_max);
  cudaError_t e = launch_unpack_records(records, num_parts, rows, k_max, parts, stream);
  if (e == cudaSuccess) {
    Traced tr(kTraceMerge, stream);
    e = launch_merge(rows, num_parts, V, k_max, parts, sel_ids, row_k, lse, sel_logprob, topk_ids, topk_logprobs,
                     dev_status, stream, /*pdl=*/true, nullptr, sms);
  }
  return from_cuda(e);
}

lmh_status lmh_debug_set_wait_limit(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns == 0 ? 2000000000ull : limit_ns, std::memory_order_relaxed);
  return LMH_OK;
}

lmh_status lmh_trace_enable(int32_t enable) {
  g_trace_on = enable != 0;
  return LMH_OK;
}

lmh_status lmh_trace_read(const char* kernel, int64_t* launches, double* total_ms) {
  if (!kernel || !launches || !total_ms) return LMH_ERR_INVALID_ARG;
  const lmh_status st = trace_drain();
  for (int k = 0; k < kTraceCount; ++k) {
    if (std::strcmp(kernel, kTraceNames[k]) == 0) {
      std::lock_guard<std::mutex> lock(g_trace_mu);
      *launches = g_trace_launches[k];
      *total_ms = g_trace_ms[k];
      return st;
    }
  }
  return LMH_ERR_INVALID_ARG;
}

void lmh_trace_reset(void) {
  trace_drain();
  std::lock_guard<std::mutex> lock(g_trace_mu);
  for (int k = 0; k < kTraceCount; ++k) {
    g_trace_launches[k] = 0;
    g_trace_ms[k] = 0.0;
  }
}

}  // extern "C"
