/*
 * lmh.h -- C ABI of liblmh, the LM-head logprob library for one NVIDIA GB300
 * GPU (sm_103a).
 *
 * The library computes the output-head hot path of LLM serving:
 *
 *   1. lmh_select_rows          pick the rows of a packed batch that are
 *                               sampled and emit compacted prefix sums;
 *   2. lmh_project_logprobs     gather those rows, project them through the
 *                               [hidden x vocab] head on the tensor cores and
 *                               reduce every row over the full vocabulary to
 *                               an O(k+1) result without writing the
 *                               [rows x vocab] logits to memory;
 *   3. lmh_logprobs_from_logits the same reduction for logits that already
 *                               exist (prompt scoring of logits chunks).
 *
 * lmh_project_partials and lmh_merge_records split step 2 over GPUs that each
 * hold a share of the vocabulary (a vocabulary-parallel head).
 *
 * The O(k+1) result of a row is: lse (fp32 log-sum-exp over the vocabulary),
 * the selected token's logprob, and the exact top-k (ids and logprobs),
 * sorted by logit descending with exact ties ordered by ascending token id.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named "device" are device memory owned by the caller (for
 *   example PyTorch tensors).  The library allocates no memory per call and
 *   keeps no per-call state; scratch memory is the caller's `workspace`.
 * - Every call is enqueued on `stream` and returns without waiting for the
 *   GPU: no host synchronisation and no device->host copy happens inside.
 * - Kernels are launched with programmatic dependent launch, so a call's
 *   first kernel may start while the kernel enqueued before it finishes.
 *   Before it waits for that kernel it reads only the head weights W (projection
 *   entry points) or the logits and selected ids of its first chunks (logits
 *   entry points).  Those inputs must therefore not be written by a kernel
 *   enqueued right before the call that itself triggers programmatic dependent
 *   launch before writing them (ordinary kernels, and this library's own, do
 *   not).
 * - Host-side argument checks return an error status and launch nothing.
 *   Errors only visible on the device (bad cu_seqlens, an id out of range)
 *   set bits (LMH_DS_*) in the caller's optional `dev_status` word with an
 *   atomic OR; kernels never trap.  The caller zeroes that word.
 * - Matrices are row-major; `*_stride` arguments are in elements.
 * - The first call on a device performs a one-time set-up (kernel attributes,
 *   driver entry points) under a once-flag.
 */
#ifndef LMH_H
#define LMH_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LMH_VERSION 1

/* Largest k (top-k entries per row) any entry point accepts. */
#define LMH_K_MAX 128
/* k_max = LMH_K_FULL asks for the full-vocabulary output: topk_logprobs
 * receives [rows x V] logprobs in token-id order and topk_ids is not written
 * (openinfer issue #719, "Acceptance criteria": the -1 behaviour is the
 * frontend's full-vocabulary contract). */
#define LMH_K_FULL (-1)

typedef enum lmh_status {
    LMH_OK = 0,
    LMH_ERR_INVALID_ARG = 1,         /* null required pointer, bad size, k > vocab, ... */
    LMH_ERR_UNSUPPORTED = 2,         /* valid request this version does not implement    */
    LMH_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < lmh_workspace_bytes(...)       */
    LMH_ERR_CUDA = 4,                /* a CUDA runtime/driver call failed                 */
    LMH_ERR_TIMEOUT = 5              /* reserved: device waits report LMH_DS_TIMEOUT      */
} lmh_status;

typedef enum lmh_dtype { LMH_BF16 = 0, LMH_F16 = 1, LMH_F32 = 2 } lmh_dtype;

/* Storage of the head weight W, whose math shape is [H x V]. */
typedef enum lmh_w_layout {
    LMH_W_VH = 0, /* stored [V x H] row-major: PyTorch lm_head.weight (H contiguous) */
    LMH_W_HV = 1  /* stored [H x V] row-major (V contiguous; V % 8 == 0)            */
} lmh_w_layout;

/* Which entry point a workspace is sized for. */
typedef enum lmh_path { LMH_PATH_PROJECT = 0, LMH_PATH_FROM_LOGITS = 1, LMH_PATH_PROBE = 2 } lmh_path;

/* Device status bits (OR-ed into *dev_status). */
#define LMH_DS_BAD_CU_SEQLENS 0x1u       /* cu[0] != 0, cu decreasing, or an empty prefill segment */
#define LMH_DS_SEL_OUT_OF_RANGE 0x2u     /* a selected id outside [0, V) other than -1 (row gets NaN) */
#define LMH_DS_ROWS_OVERFLOW 0x4u        /* more selected rows than max_out_rows (extra rows dropped) */
#define LMH_DS_ROW_IDX_OUT_OF_RANGE 0x8u /* a row index outside [0, num_tokens) (row reads zeros)   */
#define LMH_DS_TIMEOUT 0x10u             /* a bounded device-side wait gave up (kernel returned)     */
#define LMH_DS_NO_ALLOWED_TOKEN 0x20u    /* sampling: a row's mask allows no token (id -1, NaN)      */

/*
 * lmh_select_rows -- which rows of a packed batch are sampled.
 *
 * Defined by the vllm-metal release v0.4.0.dev20260831, "Summary": decode
 * rows are kept; prefill segment j is sampled at its last row,
 * cu_seqlens[num_decode + j + 1] - 1; pure-decode steps are unchanged; since
 * logits are no longer row-aligned with the input, compacted prefix sums
 * (logits_cu_seqlens) are emitted while cu_seqlens itself stays valid for
 * other consumers.  Readings where the page is silent: a decode sequence of
 * several rows keeps all of them; all_rows_mask[s] != 0 keeps every row of
 * prefill segment s (prompt scoring of every position, openinfer issue #719,
 * "Description").
 *
 *   cu_seqlens        device int32 [num_seqs + 1], cu[0] = 0, non-decreasing.
 *   num_seqs          number of sequences S (>= 0).
 *   num_decode        sequences [0, num_decode) are decode sequences.
 *   all_rows_mask     device uint8 [num_seqs] or NULL (all zero).
 *   max_out_rows      capacity of row_idx.
 *   row_idx           device int32 [max_out_rows], out: selected rows, ascending.
 *   logits_cu_seqlens device int32 [num_seqs + 1], out: logits_cu[0] = 0,
 *                     logits_cu[s+1] = logits_cu[s] + rows taken from s.
 *   dev_status        device uint32 or NULL.
 * Bad cu_seqlens set LMH_DS_BAD_CU_SEQLENS; an offending sequence contributes
 * no row.  More than max_out_rows rows set LMH_DS_ROWS_OVERFLOW (the rows
 * beyond the capacity are dropped; logits_cu_seqlens keeps the full counts).
 * Errors: LMH_ERR_INVALID_ARG for null pointers, negative sizes or
 * num_decode > num_seqs.
 */
lmh_status lmh_select_rows(const int32_t* cu_seqlens, int32_t num_seqs, int32_t num_decode,
                           const uint8_t* all_rows_mask, int32_t max_out_rows, int32_t* row_idx,
                           int32_t* logits_cu_seqlens, uint32_t* dev_status, cudaStream_t stream);

/*
 * lmh_count_selected_rows -- host helper: the number of rows lmh_select_rows
 * selects, computed from a HOST copy of cu_seqlens / all_rows_mask, so that a
 * caller can size buffers and pass `rows` without a device synchronisation.
 * Returns -1 for an invalid batch (same rules as above).
 */
int32_t lmh_count_selected_rows(const int32_t* cu_seqlens_host, int32_t num_seqs,
                                int32_t num_decode, const uint8_t* all_rows_mask_host);

/*
 * lmh_workspace_bytes -- bytes of scratch the given entry point needs for
 * these sizes on the current device (the split of the vocabulary depends on
 * its SM count).  `hidden` is ignored for LMH_PATH_FROM_LOGITS.  Returns 0
 * for sizes the entry point rejects.  The workspace must be 256-byte aligned.
 */
size_t lmh_workspace_bytes(int32_t rows, int32_t hidden, int32_t vocab, int32_t k_max,
                           lmh_path path);

/*
 * lmh_project_logprobs -- selective head projection with a fused reduction.
 *
 * Defined by: vllm-metal release v0.4.0.dev20260831, "Summary" (gather the
 * sampled rows and run the head on those alone); mlxcel PR #1969 (the row
 * sliced before the head equals the full forward's row); MTPLX PR #532,
 * "Change" (one fp32 logsumexp per row, a 64-logit block-max prefilter for
 * the exact top-k, fp32(logit) - lse at the survivors and the scored token,
 * exact ties by ascending id); openinfer issue #719, "Suggested direction"
 * and "Acceptance criteria" (compute lse, the selected logprob and the top-k
 * on the device and return an O(k+1) result).
 *
 * For row i: A[i] = hidden[row_idx[i]] (or hidden[i] when row_idx is NULL),
 * z[i][v] = sum_h A[i][h] * W[h][v] with bf16 inputs and fp32 accumulation;
 * lse[i] = log sum_v exp(z[i][v]); sel_logprob[i] = z[i][sel] - lse[i];
 * topk_ids[i][r], topk_logprobs[i][r] for r < k_i = row_k[i] (or k_max):
 * the r-th best (z desc, id asc); ranks r >= k_i hold id -1 and -inf.
 *
 *   hidden            device bf16 [num_tokens x H], row stride hidden_row_stride
 *                     (>= H); 16-byte aligned base.
 *   num_tokens        rows of `hidden` (bounds for row_idx).
 *   row_idx           device int32 [rows] or NULL.
 *   rows, H, V        sizes; H % 8 == 0.
 *   W                 device bf16, layout w_layout, 16-byte aligned; with
 *                     LMH_W_HV, V % 8 == 0 (rows of V elements are 16-byte
 *                     multiples).  Both layouts run the same kernels at the
 *                     same speed: the [H x V] slices enter the tensor cores
 *                     vocabulary-major.
 *   sel_ids           device int32 [rows] or NULL; -1 = no selected token (NaN).
 *   row_k             device int32 [rows] or NULL (= k_max); values clamped to [0, k_max].
 *   k_max             0..LMH_K_MAX and <= V, or LMH_K_FULL.
 *   lse               device fp32 [rows], out.
 *   sel_logprob       device fp32 [rows], out (required when sel_ids != NULL).
 *   topk_ids          device int32 [rows x k_max], out (required when k_max > 0).
 *   topk_logprobs     device fp32 [rows x k_max], out (required when k_max > 0);
 *                     with k_max = LMH_K_FULL: device fp32 [rows x V], out,
 *                     16-byte aligned, entry [i][v] = fp32(z[i][v]) - lse[i]
 *                     (row_k and topk_ids are ignored).
 *   logits_out        device fp32 [rows x V] or NULL (16-byte aligned): when
 *                     given, the fp32 logits are also written (the
 *                     materializing arm and debugging); the reduction
 *                     results are unchanged.
 *   workspace         device, >= lmh_workspace_bytes(rows, H, V, k_max,
 *                     LMH_PATH_PROJECT) bytes, 256-byte aligned.
 * Errors: LMH_ERR_INVALID_ARG, LMH_ERR_UNSUPPORTED (k_max < -1 or > LMH_K_MAX,
 * LMH_W_HV with V % 8 != 0, H % 8 != 0, misaligned pointers),
 * LMH_ERR_WORKSPACE_TOO_SMALL, LMH_ERR_CUDA.  Device: LMH_DS_SEL_OUT_OF_RANGE,
 * LMH_DS_ROW_IDX_OUT_OF_RANGE, LMH_DS_TIMEOUT.
 */
lmh_status lmh_project_logprobs(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                const int32_t* row_idx, int32_t rows, int32_t H, const void* W,
                                lmh_w_layout w_layout, int32_t V, const int32_t* sel_ids,
                                const int32_t* row_k, int32_t k_max, float* lse,
                                float* sel_logprob, int32_t* topk_ids, float* topk_logprobs,
                                float* logits_out, void* workspace, size_t workspace_bytes,
                                uint32_t* dev_status, cudaStream_t stream);

/*
 * lmh_project_logprobs_scaled -- lmh_project_logprobs with a head transform.
 *
 * Defined by: vllm-metal release v0.4.0.dev20260831, "Summary": some models
 * scale their head output (Cohere's logit_scale multiplies the logits,
 * Granite's logits_scaling divides them), and a head reproduced without the
 * scale gives silently wrong logits.  Here every logit is
 * fp32(logit_scale * (A . W)) before the reduction (and in logits_out):
 * pass logit_scale = s for Cohere, 1 / d for Granite's logits_scaling = d.
 *
 *   logit_scale       finite and > 0 (LMH_ERR_INVALID_ARG otherwise); 1 is
 *                     lmh_project_logprobs itself.
 * Every other argument, result and error as lmh_project_logprobs.
 */
lmh_status lmh_project_logprobs_scaled(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                       const int32_t* row_idx, int32_t rows, int32_t H, const void* W,
                                       lmh_w_layout w_layout, int32_t V, const int32_t* sel_ids,
                                       const int32_t* row_k, int32_t k_max, float* lse, float* sel_logprob,
                                       int32_t* topk_ids, float* topk_logprobs, float* logits_out,
                                       void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                       float logit_scale, cudaStream_t stream);

/*
 * Device-side sampling (lmh_project_logprobs_sample), Gumbel-max over the
 * allowed tokens of each row; the grammar bitmask is given per selected row
 * (the compacted layout: vllm-metal release v0.4.0.dev20260831, "Testing",
 * bitmask application under the compacted layout).
 *
 * For row i, with z the (scaled) fp32 logits of lmh_project_logprobs:
 *   allowed(v)  = allowed_mask is NULL, or bit (v % 32) of
 *                 allowed_mask[i * mask_words + v / 32] is set;
 *   T           = temperature[i] (1 when temperature is NULL);
 *   score(v)    = z[i][v] / T + g(v) for T > 0, z[i][v] for T <= 0 (greedy);
 *   g(v)        = -log(-log u), u = ((w >> 9) + 0.5) * 2^-23, w = word (v & 3)
 *                 of Philox4x32-10 (Salmon et al., SC 2011) with counter
 *                 (v >> 2, lo(off), hi(off), 0x53414D50), key (lo(seed),
 *                 hi(seed)), off = offsets[i] (i when offsets is NULL);
 *   sampled_ids[i] = the allowed v with the largest score, ties to the
 *                 smaller id; -1 when no token is allowed (and
 *                 LMH_DS_NO_ALLOWED_TOKEN is set);
 *   sampled_logprob[i] = z[i][sampled] - lse[i] (the unmasked, untempered
 *                 distribution); NaN for -1.
 * The noise is computed with fast fp32 logarithms; a draw can differ from an
 * exact-arithmetic draw only when two scores are within the fp32 rounding of
 * the head and the noise.
 */
typedef struct lmh_sampling {
  const float* temperature;     /* device fp32 [rows] or NULL */
  const uint32_t* allowed_mask; /* device u32 [rows x mask_words] or NULL */
  int32_t mask_words;           /* >= ceil(V / 32) when allowed_mask is given */
  uint64_t seed;
  const int64_t* offsets;       /* device int64 [rows] or NULL */
  int32_t* sampled_ids;         /* device int32 [rows], out (required) */
  float* sampled_logprob;       /* device fp32 [rows], out, or NULL */
} lmh_sampling;

/*
 * lmh_project_logprobs_sample -- lmh_project_logprobs_scaled plus the
 * sampled token of every row (the same pass over W).  sampling may not be
 * NULL; its pointers are all device memory owned by the caller.
 * Errors: as lmh_project_logprobs_scaled, and LMH_ERR_INVALID_ARG for a
 * NULL sampling or sampled_ids, or mask_words < ceil(V / 32) with a mask.
 */
lmh_status lmh_project_logprobs_sample(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                       const int32_t* row_idx, int32_t rows, int32_t H, const void* W,
                                       lmh_w_layout w_layout, int32_t V, const int32_t* sel_ids,
                                       const int32_t* row_k, int32_t k_max, float* lse, float* sel_logprob,
                                       int32_t* topk_ids, float* topk_logprobs, float* logits_out,
                                       void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                       float logit_scale, const lmh_sampling* sampling, cudaStream_t stream);

/*
 * lmh_probe_selective -- does this library's selective head reproduce the
 * model's own head output?
 *
 * Defined by: vllm-metal release v0.4.0.dev20260831, "Summary"
 * (supports_selective_logits probes once at load and demands bit-exact
 * equality with the model's own output; on a mismatch the engine keeps full
 * logits) and "Testing" (the probe rejects a model that scales its head
 * output when the scale is not reproduced).
 *
 *   hidden, hidden_row_stride, num_tokens, row_idx, rows, H, W, V:
 *                     as lmh_project_logprobs (row_idx = the rows to probe).
 *   logit_scale       the head transform to reproduce (1 = none; > 0).
 *   ref_logits        device f32 [rows x V] (row stride V): the model's own
 *                     logits of those rows.
 *   tolerance         an element mismatches when |ours - ref| > tolerance or
 *                     exactly one of them is NaN; 0 asks for bit-exact values
 *                     (except that +0 and -0 match).
 *   mismatches        device u32, out: the number of mismatching elements
 *                     (written, not accumulated).
 *   workspace         >= lmh_workspace_bytes(rows, H, V, 0, LMH_PATH_PROBE)
 *                     bytes, 256-byte aligned.
 * Errors: as lmh_project_logprobs, and LMH_ERR_INVALID_ARG for a null
 * ref_logits or mismatches, a negative or NaN tolerance, or a logit_scale
 * that is not finite and > 0.
 */
lmh_status lmh_probe_selective(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                               const int32_t* row_idx, int32_t rows, int32_t H, const void* W, int32_t V,
                               float logit_scale, const float* ref_logits, float tolerance,
                               uint32_t* mismatches, void* workspace, size_t workspace_bytes,
                               uint32_t* dev_status, cudaStream_t stream);

/*
 * lmh_logprobs_from_logits -- the same per-row reduction for logits that are
 * already in device memory (prompt scoring of logits chunks).
 *
 * Defined by MTPLX PR #532, "Summary" and "Change" (per 256-row chunk of
 * 248,320 logits: one fp32 logsumexp per row; top-k through the 64-logit
 * block-max prefilter that keeps the k blocks with the largest maxima and
 * selects the exact top-k among their entries; fp32(logit) - lse only at the
 * survivors and the scored token; exact ties by ascending id) and openinfer
 * issue #719 (reusable for decode rows and batches of prompt positions).
 *
 *   logits            device [rows x V] of dtype, row stride row_stride (>= V),
 *                     base aligned to sizeof(dtype).  When the base, the
 *                     row stride and the row length are multiples of 16
 *                     bytes the logits are streamed with bulk copies, else
 *                     with plain loads.
 *   sel_ids, row_k, k_max, lse, sel_logprob, topk_ids, topk_logprobs:
 *                     as for lmh_project_logprobs (logit = the given value
 *                     widened exactly to fp32).
 *   workspace         >= lmh_workspace_bytes(rows, 0, V, k_max,
 *                     LMH_PATH_FROM_LOGITS) bytes, 256-byte aligned.
 * Results for NaN or +inf logits are unspecified.  A row of only -inf gives
 * lse = -inf and NaN logprobs (ids 0..k-1).
 * Errors: as lmh_project_logprobs.
 */
lmh_status lmh_logprobs_from_logits(const void* logits, lmh_dtype dtype, int32_t rows, int32_t V,
                                    int64_t row_stride, const int32_t* sel_ids,
                                    const int32_t* row_k, int32_t k_max, float* lse,
                                    float* sel_logprob, int32_t* topk_ids, float* topk_logprobs,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                    cudaStream_t stream);

/*
 * lmh_logprobs_from_logits_static -- lmh_logprobs_from_logits without a
 * caller workspace.
 *
 * The pages have no counterpart for this entry point.  It serves callers
 * that cannot allocate device memory when they need the reduction:
 * - an engine that gave all free HBM to its KV-cache pool at start-up;
 * - plain C code without access to the framework's allocator;
 * - a latency-critical loop where cudaMalloc/cudaFree would synchronise the
 *   device.
 * It runs the same kernels and returns the same results as
 * lmh_logprobs_from_logits. Instead of a caller workspace, it keeps its
 * partials in a fixed 8 MiB array in the library's own device memory, which
 * every GPU that loads the library holds until the process exits.  The call
 * allocates nothing.
 *
 * Arguments, results and errors are those of lmh_logprobs_from_logits,
 * minus workspace/workspace_bytes, with two differences:
 * - sizes whose partials need more than the 8 MiB are rejected with
 *   LMH_ERR_WORKSPACE_TOO_SMALL, and nothing is launched.  The partials take
 *   about rows * (4 * ceil(V / 64) + 8 * slots + 8) bytes, with slots =
 *   4 * ceil(ceil(V / 64) / 64) (whatever k_max and dtype): 256 rows x
 *   248320 need about 4.5 MB and fit; the largest batch is 479 rows at
 *   V = 248320 and 782 rows at V = 151936.
 * - the first call on each device does a one-time set-up with that device
 *   current: kernel attributes, and the array's device address via
 *   cudaGetSymbolAddress.  Make that first call before any stream capture.
 * Every call shares the one array, which keeps the previous call's contents.
 * Nothing in it needs to start at zero, but calls that overlap on the GPU
 * race on it: serialise them, on one stream or with events.
 */
lmh_status lmh_logprobs_from_logits_static(const void* logits, lmh_dtype dtype, int32_t rows,
                                           int32_t V, int64_t row_stride, const int32_t* sel_ids,
                                           const int32_t* row_k, int32_t k_max, float* lse,
                                           float* sel_logprob, int32_t* topk_ids,
                                           float* topk_logprobs, uint32_t* dev_status,
                                           cudaStream_t stream);

/*
 * Vocabulary-parallel head: several GPUs, each holding a share of the head's
 * vocabulary, together compute the same O(k+1) result as lmh_project_logprobs.
 *
 * Defined by openinfer issue #719, "Suggested direction" (a numerically sound
 * multi-stage reduction: per-part max and sum of exponentials combine exactly
 * into the log-sum-exp) and MTPLX PR #532, "Change" (the exact top-k of a row
 * lies among the union of the parts' own top-k lists; exact ties by ascending
 * token id).  Each rank calls lmh_project_partials on its share, the ranks
 * all-gather their records (any collective that concatenates equal-sized byte
 * buffers in rank order, e.g. an NCCL all-gather into the caller's device
 * memory), and every rank (or one) calls lmh_merge_records on the gathered
 * buffer.  The library itself makes no collective call.
 *
 * A record is lmh_record_bytes(k_max) bytes per row, 8-byte aligned:
 *   float m            the share's largest logit of the row (-inf: none)
 *   float s            sum over the share of exp(logit - m)
 *   float sel_logit    the selected token's logit, when it lies in the share
 *   uint32 flags       bit 0: sel_logit is set
 *   uint64 keys[k_max] the share's best k entries, best first: a key is
 *                      (order-preserving bits of the fp32 logit << 32) |
 *                      ~token_id, with global token ids; 0 = no entry.
 */
size_t lmh_record_bytes(int32_t k_max);

/*
 * lmh_project_partials -- one share of a vocabulary-parallel head.
 *
 * As lmh_project_logprobs (same hidden / row_idx / rows / H / sel_ids /
 * row_k / k_max meanings, the same fp32 accumulation and the same per-row
 * reduction), over the share's tokens [v_begin, v_begin + v_count) only:
 *   W_share    device bf16 [v_count x H], rows v_begin.. of lm_head.weight
 *              (LMH_W_VH; other layouts: LMH_ERR_UNSUPPORTED).
 *   V          the full vocabulary (sel_ids and returned ids are global).
 *   records    device [rows] records (lmh_record_bytes(k_max) each), out.
 *   workspace  >= lmh_workspace_bytes(rows, H, v_count, k_max, LMH_PATH_PROJECT).
 * k_max in [0, LMH_K_MAX] and <= v_count.  No logits are written.
 * Errors: as lmh_project_logprobs; LMH_ERR_INVALID_ARG also when the share is
 * empty or leaves [0, V).
 */
lmh_status lmh_project_partials(const void* hidden, int64_t hidden_row_stride, int32_t num_tokens,
                                const int32_t* row_idx, int32_t rows, int32_t H, const void* W_share,
                                lmh_w_layout w_layout, int32_t v_begin, int32_t v_count, int32_t V,
                                const int32_t* sel_ids, const int32_t* row_k, int32_t k_max, void* records,
                                void* workspace, size_t workspace_bytes, uint32_t* dev_status,
                                cudaStream_t stream);

/* Workspace of lmh_merge_records (bytes; 0 for invalid arguments). */
size_t lmh_merge_workspace_bytes(int32_t rows, int32_t num_parts, int32_t k_max);

/*
 * lmh_merge_records -- the rows' final results from the gathered records.
 *
 *   records     device [num_parts][rows] records, part p's rows contiguous
 *               (the layout of an all-gather of each rank's record buffer).
 *               The parts' shares must partition [0, V).
 *   V, sel_ids, row_k, k_max, lse, sel_logprob, topk_ids, topk_logprobs:
 *               as for lmh_project_logprobs (k_max must equal the k_max the
 *               records were made with).
 *   workspace   >= lmh_merge_workspace_bytes(rows, num_parts, k_max).
 * lse = M + log(sum_p s_p exp(m_p - M)), M = max_p m_p; the top-k is the best
 * k keys of the parts' lists; logprob = logit - lse.
 * Errors: as lmh_project_logprobs.
 */
lmh_status lmh_merge_records(const void* records, int32_t num_parts, int32_t rows, int32_t V,
                             const int32_t* sel_ids, const int32_t* row_k, int32_t k_max, float* lse,
                             float* sel_logprob, int32_t* topk_ids, float* topk_logprobs, void* workspace,
                             size_t workspace_bytes, uint32_t* dev_status, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
const char* lmh_status_string(lmh_status status);

/* LMH_VERSION of the loaded library. */
int32_t lmh_version(void);

/*
 * Kernel tracing (device time per kernel, measured with CUDA events recorded
 * on the launching stream around every launch while enabled).  Not for use
 * while a stream is being captured into a CUDA graph.
 *
 * lmh_trace_enable(1) starts recording, lmh_trace_enable(0) stops.
 * lmh_trace_read waits for the recorded events, then reports the launches
 * and total milliseconds of the named kernel ("select_rows", "gather_rows",
 * "head_logprobs", "merge_partials", "logits_reduce" (the streaming pass of
 * lmh_logprobs_from_logits), "logits_select" (its per-row selection),
 * "full_logprobs" (the pass that writes the k_max = LMH_K_FULL output)) since
 * the last reset.
 * lmh_trace_reset clears the totals.
 */
lmh_status lmh_trace_enable(int32_t enable);
lmh_status lmh_trace_read(const char* kernel, int64_t* launches, double* total_ms);
void lmh_trace_reset(void);

/*
 * lmh_debug_set_wait_limit -- test hook for the timeout path; not for
 * production use.  The pages have no counterpart.
 *
 * Inside a kernel, every wait on another role of the same CTA (a shared-memory
 * stage, an accumulator, a chunk) gives up after this limit: the kernel sets
 * LMH_DS_TIMEOUT in *dev_status, stops its loops, lets its copies and tensor-
 * core work in flight finish (those drain waits keep a fixed 2 s limit), frees
 * its tensor memory and returns, so the context stays usable.  The default is
 * 2 s, far above any legitimate wait; a test sets a limit shorter than the
 * latency of one load so that the first wait runs out, then calls with 0 to
 * restore the default.  The value applies to kernels launched after the call,
 * from any thread.  Always LMH_OK.
 */
lmh_status lmh_debug_set_wait_limit(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* LMH_H */
