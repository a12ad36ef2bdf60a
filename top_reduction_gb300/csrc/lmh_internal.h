// lmh_internal.h -- host-side interfaces between the C ABI (lmh_api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "lmh.h"

namespace lmh {

constexpr int kBlock = 64;  // logits per prefilter block (MTPLX PR #532, "Change")

// Work split of the standalone reduction: the flattened (row, 64-block) space
// is cut into n_ranges equal ranges of `per` blocks; a row meets at most
// `splits` ranges, which is the number of partial slots per row.  The ranges
// a row meets are [(row*nblk)/per, (row*nblk + nblk - 1)/per].
struct VocabSplit {
  int splits;    // row pieces per row, at most
  int per;       // 64-blocks per range
  int n_ranges;  // ranges in total
  int grid;      // persistent CTAs of the register-path stream kernel (one range each)
  int ctas;      // persistent CTAs of the TMA-path stream kernel (four per SM)
  int nblk;      // 64-blocks per row
  int slots;     // (m, s) slots per row in the workspace (enough for either stream kernel)
};

// The chunk counter of the standalone reduction's dynamic schedule.  It is never
// reset: after every call the select kernel records its value as the next call's
// base, with the bitwise complement as a check.  A stream kernel that finds the
// pair consistent draws chunks base + 0, 1, ...; one that does not (a workspace
// never used by this path, or reused for something else) hands out its chunks in
// a fixed order instead (the same results, a little slower).
struct TicketState {
  unsigned long long ticket;
  unsigned long long base;
  unsigned long long check;  // ~base when base is valid
};

// Per-(row, split) partial results, laid out in the caller's workspace:
//   part_ms   float2 [rows * splits]            (chunk max m, sum exp(x - m))
//   part_keys uint64 [rows * splits * k_max]    sorted top-k keys of the chunk
//   sel_logit float  [rows]                     logit of the selected token
struct Partials {
  float2* part_ms;
  unsigned long long* part_keys;
  float* sel_logit;
  struct TicketState* ticket;  // standalone reduction: the dynamic chunk schedule's counter (else unused)
  float4* part_samp;     // head path: per-(row, split) sampling partial (best score, id bits, z, -)
  float* bmax;  // standalone reduction: block maxima [rows * nblk] (else unused)
};

// Device-side sampling on the head path (lmh_project_logprobs_sample): Gumbel-max
// over the allowed tokens, Philox4x32-10 noise keyed by (seed, row offset, token).
struct SampleArgs {
  int enabled;
  const float* temperature;  // [rows] or null (1); <= 0: greedy
  const uint32_t* mask;      // [rows x mask_words] allowed-token bits, or null (all allowed)
  int mask_words;
  uint64_t seed;
  const int64_t* offsets;  // [rows] counter offsets, or null (the row index)
  int32_t* ids_out;        // [rows]
  float* lp_out;           // [rows] z[id] - lse, or null
};

// Vocabulary-parallel head: one rank's result for one row over its share of the
// vocabulary, as exchanged between ranks (include/lmh.h, lmh_record_bytes):
// the share's max m and sum exp(z - m), the selected token's logit when the
// token lies in the share (flags bit 0), then k_max sortable keys, best first,
// with global token ids (0: no entry).
struct VocabRecord {
  float m;
  float s;
  float sel_logit;
  uint32_t flags;
};
constexpr uint32_t kRecordHasSel = 1u;
__host__ __device__ inline size_t record_bytes(int k_max) {
  return sizeof(VocabRecord) + 8 * static_cast<size_t>(k_max > 0 ? k_max : 0);
}

// Where the merge writes a vocabulary-parallel record instead of final results.
struct RecordOut {
  unsigned char* base;  // [rows] records of record_bytes(k_max)
  int v_begin, v_count;  // the share: token ids [v_begin, v_begin + v_count)
};

// Final per-row results (the outputs of lmh_project_logprobs / lmh_logprobs_from_logits).
struct RowOutputs {
  float* lse;
  float* sel_logprob;
  int32_t* topk_ids;
  float* topk_logprobs;
};

size_t partials_bytes(int rows, int splits, int k_max);
Partials carve_partials(void* base, int rows, int splits, int k_max);

// Limit of the kernels' bounded waits on another role of their own CTA (2 s;
// lmh_debug_set_wait_limit changes it for tests of the timeout path).
uint64_t wait_limit_ns();

// One-time per-device set-up (kernel attributes).  Returns cudaSuccess or the error.
cudaError_t logits_reduce_setup();
cudaError_t merge_setup();
cudaError_t head_setup();

VocabSplit logits_reduce_split(int rows, int V, int k_max, int num_sms);

cudaError_t launch_select_rows(const int32_t* cu, int num_seqs, int num_decode, const uint8_t* mask,
                               int max_out, int32_t* row_idx, int32_t* logits_cu, uint32_t* dev_status,
                               cudaStream_t stream);

// Workspace of the standalone reduction: part_ms [rows * slots], sel_logit
// [rows], bmax [rows * nblk], the chunk counter.
size_t stream_partials_bytes(int rows, const VocabSplit& vs);
Partials carve_stream_partials(void* base, int rows, const VocabSplit& vs);

// Ticket reset and the bulk-copy stream kernel (16-byte aligned rows), or the
// register-path stream kernel; then the per-row select kernel, which writes the
// outputs.
cudaError_t launch_logits_reduce(const void* logits, lmh_dtype dtype, int64_t row_stride, int rows, int V,
                                 VocabSplit split, const int32_t* sel, const int32_t* row_k, int k_max,
                                 Partials parts, float* lse, float* sel_logprob, int32_t* topk_ids,
                                 float* topk_logprobs, uint32_t* dev_status, cudaStream_t stream);

// Merges the `splits` partial slots of every row (head path).
cudaError_t launch_merge(int rows, int splits, int V, int k_max, Partials parts, const int32_t* sel,
                         const int32_t* row_k, float* lse, float* sel_logprob, int32_t* topk_ids,
                         float* topk_logprobs, uint32_t* dev_status, cudaStream_t stream, bool pdl = false,
                         const SampleArgs* samp = nullptr, int num_sms = 0, const RecordOut* rec = nullptr);

// Scatters the gathered records [num_parts][rows] into the merge's partials
// (one slot per part): (m, s), keys, and the selected logit from the part that holds it.
cudaError_t launch_unpack_records(const void* records, int num_parts, int rows, int k_max, Partials parts,
                                  cudaStream_t stream);

// Full-vocabulary output: out[r][v] = fp32(x[r][v]) - lse[r] (x may alias out for f32).
cudaError_t launch_full_logprobs(const void* x, lmh_dtype dtype, int64_t row_stride, int rows, int V, const float* lse,
                                 float* out, cudaStream_t stream);

// Counts the elements of ours / ref [n] that differ by more than tol (probe.cu).
cudaError_t launch_probe_compare(const float* ours, const float* ref, int64_t n, float tol, uint32_t* count,
                                 int num_sms, cudaStream_t stream);

// ---- head projection (head_gemm.cu) ----

// Tile scheduling of the fused head kernel.
struct HeadPlan {
  int m_tiles;          // ceil(rows / 128)
  int n_tiles;          // ceil(V / 256)
  int splits;           // vocabulary ranges per row (units = m_tiles * splits)
  int tiles_per_split;  // n-tiles per range
  int grid;             // persistent CTAs
  int kcap;             // per-row candidate capacity variant (1, 5, 8, 16, 20, 32 or 128)
};

HeadPlan head_plan(int rows, int H, int V, int k_max, int num_sms);

cudaError_t launch_gather_rows(const void* hidden, int64_t hidden_stride, int num_tokens,
                               const int32_t* row_idx, int rows, int H, void* out, uint32_t* dev_status,
                               cudaStream_t stream);

// final_out != nullptr (a plan with one vocabulary split): every row lies in
// one CTA's unit, so the kernel writes the final results itself and no merge
// follows; otherwise it writes the per-split partials.
cudaError_t launch_head(const void* A, int64_t a_stride, int rows, int H, const void* W, int V,
                        const HeadPlan& plan, const int32_t* sel, const int32_t* row_k, int k_max,
                        Partials parts, float* logits_out, uint32_t* dev_status, cudaStream_t stream,
                        bool pdl = false, const RowOutputs* final_out = nullptr, float logit_scale = 1.0f,
                        const SampleArgs* samp = nullptr, bool w_hv = false, int id_off = 0);

// Launch `kernel` on `stream`; with pdl = true it carries the programmatic
// stream serialization attribute, so it may start while its predecessor in the
// stream finishes (the kernel calls pdl_wait() before reading that
// predecessor's output).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- tracing (lmh_api.cu) ----
enum TraceKernel {
  kTraceSelect = 0,
  kTraceGather,
  kTraceHead,
  kTraceReduce,
  kTraceMerge,
  kTraceLogitsSelect,
  kTraceFull,
  kTraceCount
};
void trace_begin(TraceKernel k, cudaStream_t s);
void trace_end(TraceKernel k, cudaStream_t s);

}  // namespace lmh
