/*
 * oracle.c -- plain CPU reference for the LM-head logprob path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library in top_reduction_gb300/;
 * neither side includes or calls the other.
 *
 * It computes the plain definitions, in double precision, with no blocking,
 * fusion or reordering beyond what each definition states:
 *
 *   oracle_select_rows  -- which packed rows are sampled, and the compacted
 *       prefix sums.  vllm-metal release v0.4.0.dev20260831, "Summary":
 *       one row per prefill segment j, namely cu_seqlens[num_decode+j+1]-1;
 *       decode rows are all kept; logits are no longer row-aligned with the
 *       input, so a compacted logits_cu_seqlens is emitted.
 *   oracle_project      -- z[i][v] = sum_h A[i][h] * W[h][v] in f64.
 *       vllm-metal release, "Summary" (the head is a [hidden x vocab]
 *       matmul over the gathered rows); mlxcel PR #1969 (the row that is
 *       sliced before the head equals the full forward's row).
 *   oracle_logprobs     -- full-vocabulary log-softmax in f64, then a full
 *       sort by (logit descending, token id ascending).  openinfer issue
 *       #719, "Description": a full-vocabulary max pass, an f64 exp-sum pass,
 *       then a top-k pass; MTPLX PR #532, "Change": logprob = logit - lse
 *       at the survivors and at the scored token, exact ties listed by
 *       ascending token id.
 *   oracle_philox4x32_10 -- the counter-based generator Philox4x32 with
 *       10 rounds, from its published definition (Salmon, Moraes, Dror,
 *       Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
 *       per round, two 32x32->64 products of counter words with the round
 *       multipliers, the high halves XORed with the other counter words and
 *       the key, the key bumped by the Weyl constants.
 *   oracle_sample       -- Gumbel-max sampling: the token maximising
 *       z / T + g over the allowed tokens (g = -log(-log u) Gumbel noise,
 *       u uniform in (0, 1) from Philox keyed by (seed, row offset, token));
 *       T <= 0 is greedy (argmax z).  No page defines it: it is the NEXT
 *       item "device-side sampling in the head epilogue" with the grammar
 *       bitmask applied in the compacted layout (vllm-metal release,
 *       "Testing": bitmask application under the compacted layout).
 *
 * Readings where the pages are silent:
 *   - decode sequences keep all their rows [cu[s], cu[s+1]);
 *   - an empty prefill segment, a non-monotone cu_seqlens or cu[0] != 0
 *     is rejected (return code ORACLE_ERR_BAD_CU);
 *   - all_rows_mask[s] != 0 keeps every row of prefill segment s
 *     (prompt scoring of every position);
 *   - a whole row of -inf gives lse = -inf and NaN logprobs (-inf - -inf),
 *     top-k ids 0..k-1;
 *   - a selected id of -1 means "no selected token" and gives NaN; any other
 *     id outside [0, V) is rejected (ORACLE_ERR_SEL_RANGE);
 *   - ranks at or beyond a row's own k (row_k) are padded with id -1 and
 *     logprob -inf;
 *   - -0.0 and +0.0 compare equal (an exact tie, ordered by id).
 *
 * Mutation hooks: oracle_set_mutation() plants one deliberate mistake so that
 * the test suite can show that its pins catch it.  The default (0) is the
 * correct oracle; nothing but the pin-strength tests sets another value.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_BAD_CU 2
#define ORACLE_ERR_OVERFLOW 3
#define ORACLE_ERR_SEL_RANGE 4
#define ORACLE_ERR_NOMEM 5

/* dtype codes of oracle_logprobs' input */
#define ORACLE_BF16 0
#define ORACLE_F16 1
#define ORACLE_F32 2
#define ORACLE_F64 3

/* planted mistakes for the pin-strength tests (0 = none) */
#define MUT_NONE 0
#define MUT_SELECT_SHIFT 1      /* prefill row cu[s+1] instead of cu[s+1]-1  */
#define MUT_PROJECT_DROP_TERM 2 /* sum over h < H-1                          */
#define MUT_PROJECT_TRANSPOSE 3 /* read W[v][h] as if it were W[h][v]         */
#define MUT_LSE_DROP_TERM 4     /* exp-sum over v < V-1                       */
#define MUT_LOGPROB_SIGN 5      /* lse - x instead of x - lse                 */
#define MUT_TIE_ID_DESC 6       /* exact ties by descending id                */
#define MUT_TOPK_SKIP_FIRST 7   /* rank j reports sorted entry j+1            */
#define MUT_DECODE_LAST_ONLY 8  /* decode sequences keep only their last row  */
#define MUT_PHILOX_9_ROUNDS 9   /* Philox with 9 rounds                       */
#define MUT_GUMBEL_SIGN 10      /* g = +log(-log u)                           */
#define MUT_MASK_IGNORED 11     /* disallowed tokens can be sampled           */
#define MUT_TEMP_TIMES 12       /* z * T instead of z / T                     */

static int g_mutation = MUT_NONE;

void oracle_set_mutation(int m) { g_mutation = m; }
int oracle_get_mutation(void) { return g_mutation; }

/* ------------------------------------------------------------------ */
/* exact conversions to double                                          */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double bf16_bits_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 -> double, written out from the format definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits). */
static double f16_bits_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f | 0x400), e - 25); /* (1024+f) * 2^(e-15-10) */
    return sign ? -v : v;
}

static double load_as_f64(const void* base, int dtype, int64_t idx)
{
    switch (dtype) {
    case ORACLE_BF16: return bf16_bits_to_f64(((const uint16_t*)base)[idx]);
    case ORACLE_F16: return f16_bits_to_f64(((const uint16_t*)base)[idx]);
    case ORACLE_F32: return (double)((const float*)base)[idx];
    default: return ((const double*)base)[idx];
    }
}

static int resolve_threads(int threads)
{
    if (threads > 0) return threads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ------------------------------------------------------------------ */
/* 1. row selection                                                     */
/* ------------------------------------------------------------------ */

/*
 * Sequences s < num_decode are decode sequences: every row [cu[s], cu[s+1])
 * is sampled.  Sequence s >= num_decode is prefill segment j = s-num_decode:
 * its sampled row is cu[num_decode+j+1]-1 = cu[s+1]-1, or every row of the
 * segment when all_rows_mask[s] is set.  logits_cu[0] = 0 and
 * logits_cu[s+1] = logits_cu[s] + (rows taken from s).
 */
int oracle_select_rows(const int32_t* cu, int32_t num_seqs, int32_t num_decode,
                       const uint8_t* all_rows_mask, int32_t max_out,
                       int32_t* row_idx, int32_t* logits_cu, int32_t* n_sel)
{
    if (!cu || !row_idx || !logits_cu || !n_sel || num_seqs < 0 || num_decode < 0 ||
        num_decode > num_seqs || max_out < 0)
        return ORACLE_ERR_ARG;
    if (cu[0] != 0) return ORACLE_ERR_BAD_CU;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (cu[s + 1] < cu[s]) return ORACLE_ERR_BAD_CU;

    int32_t n = 0;
    logits_cu[0] = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t first, last; /* rows [first, last) are taken */
        int decode = s < num_decode;
        int every = decode || (all_rows_mask && all_rows_mask[s]);
        if (!decode && cu[s + 1] == cu[s]) return ORACLE_ERR_BAD_CU;
        if (every) {
            first = cu[s];
            last = cu[s + 1];
            if (decode && g_mutation == MUT_DECODE_LAST_ONLY && last > first)
                first = last - 1;
        } else {
            first = cu[s + 1] - 1;
            if (g_mutation == MUT_SELECT_SHIFT) first = cu[s + 1];
            last = first + 1;
        }
        for (int32_t r = first; r < last; ++r) {
            if (n >= max_out) return ORACLE_ERR_OVERFLOW;
            row_idx[n++] = r;
        }
        logits_cu[s + 1] = n;
    }
    *n_sel = n;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* 2. head projection in f64                                            */
/* ------------------------------------------------------------------ */

typedef struct {
    const uint16_t* hidden; /* bf16 bits, row stride hidden_stride */
    int64_t hidden_stride;
    const int32_t* row_idx; /* NULL = rows 0..rows-1 */
    int32_t rows, H, V;
    const uint16_t* W; /* bf16 bits */
    int w_layout;      /* 0: stored [V x H] (W[h][v] at v*H+h); 1: stored [H x V] */
    double* z;         /* [rows x V] */
    int64_t begin, end; /* flattened (i, v) range of this worker */
} project_job;

static void* project_worker(void* arg)
{
    project_job* j = (project_job*)arg;
    const int32_t H = j->H, V = j->V;
    double* a = (double*)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (!a) return (void*)1;
    int32_t cur_row = -1;
    for (int64_t t = j->begin; t < j->end; ++t) {
        int32_t i = (int32_t)(t / V);
        int32_t v = (int32_t)(t % V);
        if (i != cur_row) {
            int64_t src = j->row_idx ? j->row_idx[i] : i;
            const uint16_t* hrow = j->hidden + src * j->hidden_stride;
            for (int32_t h = 0; h < H; ++h) a[h] = bf16_bits_to_f64(hrow[h]);
            cur_row = i;
        }
        int32_t hend = (g_mutation == MUT_PROJECT_DROP_TERM) ? H - 1 : H;
        double acc = 0.0;
        if (g_mutation == MUT_PROJECT_TRANSPOSE) {
            /* misread the [V x H] buffer as [H x V] */
            for (int32_t h = 0; h < hend; ++h)
                acc += a[h] * bf16_bits_to_f64(j->W[(int64_t)h * V + v]);
        } else if (j->w_layout == 0) {
            const uint16_t* wcol = j->W + (int64_t)v * H; /* W[.][v] contiguous */
            for (int32_t h = 0; h < hend; ++h) acc += a[h] * bf16_bits_to_f64(wcol[h]);
        } else {
            for (int32_t h = 0; h < hend; ++h)
                acc += a[h] * bf16_bits_to_f64(j->W[(int64_t)h * V + v]);
        }
        j->z[t] = acc;
    }
    free(a);
    return NULL;
}

/*
 * z[i][v] = sum over h of A[i][h] * W[h][v], with A[i] = hidden[row_idx[i]]
 * (or hidden[i] when row_idx is NULL).  Each bf16 x bf16 product is exact in
 * f64; only the f64 running sum rounds.  Work is split over the flattened
 * (i, v) space among `threads` workers (0 = all online cores); the number
 * used is written to *threads_used.
 */
int oracle_project(const uint16_t* hidden, int64_t hidden_stride, const int32_t* row_idx,
                   int32_t rows, int32_t H, const uint16_t* W, int w_layout, int32_t V,
                   double* z, int threads, int* threads_used)
{
    if (!hidden || !W || !z || rows < 0 || H <= 0 || V <= 0 || (w_layout != 0 && w_layout != 1))
        return ORACLE_ERR_ARG;
    int64_t total = (int64_t)rows * V;
    int nt = resolve_threads(threads);
    if ((int64_t)nt > total) nt = (int)(total > 0 ? total : 1);
    if (threads_used) *threads_used = nt;
    if (total == 0) return ORACLE_OK;
    project_job* jobs = (project_job*)calloc((size_t)nt, sizeof(project_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return ORACLE_ERR_NOMEM; }
    int rc = ORACLE_OK;
    for (int k = 0; k < nt; ++k) {
        project_job* j = &jobs[k];
        j->hidden = hidden; j->hidden_stride = hidden_stride; j->row_idx = row_idx;
        j->rows = rows; j->H = H; j->V = V; j->W = W; j->w_layout = w_layout; j->z = z;
        j->begin = total * k / nt;
        j->end = total * (k + 1) / nt;
        if (pthread_create(&tids[k], NULL, project_worker, j) != 0) {
            j->end = j->begin; /* run it inline instead */
            project_worker(j);
            tids[k] = 0;
        }
    }
    for (int k = 0; k < nt; ++k) {
        void* ret = NULL;
        if (tids[k]) pthread_join(tids[k], &ret);
        if (ret) rc = ORACLE_ERR_NOMEM;
    }
    free(jobs);
    free(tids);
    return rc;
}

/* ------------------------------------------------------------------ */
/* 3. full-vocabulary log-softmax in f64 + full sort                    */
/* ------------------------------------------------------------------ */

typedef struct {
    double x;
    int32_t id;
} entry;

/* strict total order: larger logit first; exact ties by ascending id */
static int entry_cmp(const void* pa, const void* pb)
{
    const entry* a = (const entry*)pa;
    const entry* b = (const entry*)pb;
    if (a->x > b->x) return -1;
    if (a->x < b->x) return 1;
    if (g_mutation == MUT_TIE_ID_DESC) return (a->id < b->id) ? 1 : (a->id > b->id) ? -1 : 0;
    return (a->id < b->id) ? -1 : (a->id > b->id) ? 1 : 0;
}

typedef struct {
    const void* x;
    int dtype;
    int32_t V;
    int64_t row_stride;
    const int32_t* sel;   /* nullable */
    const int32_t* row_k; /* nullable = k_max */
    int32_t k_max;
    double* lse;
    double* sel_lp;
    int32_t* topk_ids;
    double* topk_lp;
    int32_t row_begin, row_end;
    int err;
} logprob_job;

static void* logprob_worker(void* arg)
{
    logprob_job* j = (logprob_job*)arg;
    const int32_t V = j->V;
    double* x = (double*)malloc(sizeof(double) * (size_t)V);
    entry* e = (entry*)malloc(sizeof(entry) * (size_t)V);
    if (!x || !e) { free(x); free(e); j->err = ORACLE_ERR_NOMEM; return NULL; }
    for (int32_t i = j->row_begin; i < j->row_end; ++i) {
        for (int32_t v = 0; v < V; ++v)
            x[v] = load_as_f64(j->x, j->dtype, (int64_t)i * j->row_stride + v);

        /* max pass */
        double m = -INFINITY;
        for (int32_t v = 0; v < V; ++v)
            if (x[v] > m) m = x[v];
        /* exp-sum pass: lse = m + log(sum exp(x - m)) */
        double lse;
        if (m == -INFINITY) {
            lse = -INFINITY;
        } else {
            int32_t vend = (g_mutation == MUT_LSE_DROP_TERM) ? V - 1 : V;
            double s = 0.0;
            for (int32_t v = 0; v < vend; ++v) s += exp(x[v] - m);
            lse = m + log(s);
        }
        j->lse[i] = lse;

        /* selected token */
        if (j->sel) {
            int32_t t = j->sel[i];
            if (t == -1) {
                j->sel_lp[i] = NAN;
            } else if (t < 0 || t >= V) {
                j->sel_lp[i] = NAN;
                j->err = ORACLE_ERR_SEL_RANGE;
            } else {
                j->sel_lp[i] = (g_mutation == MUT_LOGPROB_SIGN) ? lse - x[t] : x[t] - lse;
            }
        }

        /* top-k pass: full sort by (x desc, id asc) */
        int32_t k = j->row_k ? j->row_k[i] : j->k_max;
        if (k > j->k_max) k = j->k_max;
        if (k < 0) k = 0;
        if (j->k_max > 0) {
            for (int32_t v = 0; v < V; ++v) { e[v].x = x[v]; e[v].id = v; }
            qsort(e, (size_t)V, sizeof(entry), entry_cmp);
            int skip = (g_mutation == MUT_TOPK_SKIP_FIRST) ? 1 : 0;
            for (int32_t r = 0; r < j->k_max; ++r) {
                int64_t o = (int64_t)i * j->k_max + r;
                if (r < k && r + skip < V) {
                    const entry* pe = &e[r + skip];
                    j->topk_ids[o] = pe->id;
                    j->topk_lp[o] = (g_mutation == MUT_LOGPROB_SIGN) ? lse - pe->x : pe->x - lse;
                } else {
                    j->topk_ids[o] = -1;
                    j->topk_lp[o] = -INFINITY;
                }
            }
        }
    }
    free(x);
    free(e);
    return NULL;
}

/*
 * Per row i of x ([rows x V], row stride row_stride elements, dtype as
 * above): lse[i], sel_lp[i] (if sel != NULL), and the k_i = row_k[i] (or
 * k_max) best (logit desc, id asc) entries in topk_ids / topk_lp
 * ([rows x k_max]).  k_max may be 0 (topk outputs untouched, may be NULL).
 */
int oracle_logprobs(const void* x, int dtype, int32_t rows, int32_t V, int64_t row_stride,
                    const int32_t* sel, const int32_t* row_k, int32_t k_max, double* lse,
                    double* sel_lp, int32_t* topk_ids, double* topk_lp, int threads,
                    int* threads_used)
{
    if (!x || !lse || rows < 0 || V <= 0 || row_stride < V || k_max < 0 || k_max > V ||
        dtype < ORACLE_BF16 || dtype > ORACLE_F64 || (sel && !sel_lp) ||
        (k_max > 0 && (!topk_ids || !topk_lp)))
        return ORACLE_ERR_ARG;
    int nt = resolve_threads(threads);
    if (nt > rows) nt = rows > 0 ? rows : 1;
    if (threads_used) *threads_used = nt;
    if (rows == 0) return ORACLE_OK;
    logprob_job* jobs = (logprob_job*)calloc((size_t)nt, sizeof(logprob_job));
    pthread_t* tids = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return ORACLE_ERR_NOMEM; }
    for (int k = 0; k < nt; ++k) {
        logprob_job* j = &jobs[k];
        j->x = x; j->dtype = dtype; j->V = V; j->row_stride = row_stride; j->sel = sel;
        j->row_k = row_k; j->k_max = k_max; j->lse = lse; j->sel_lp = sel_lp;
        j->topk_ids = topk_ids; j->topk_lp = topk_lp;
        j->row_begin = (int32_t)((int64_t)rows * k / nt);
        j->row_end = (int32_t)((int64_t)rows * (k + 1) / nt);
        if (pthread_create(&tids[k], NULL, logprob_worker, j) != 0) {
            logprob_worker(j);
            tids[k] = 0;
        }
    }
    int rc = ORACLE_OK;
    for (int k = 0; k < nt; ++k) {
        if (tids[k]) pthread_join(tids[k], NULL);
        if (jobs[k].err && rc == ORACLE_OK) rc = jobs[k].err;
    }
    free(jobs);
    free(tids);
    return rc;
}

/* number of online cores, for reporting */
int oracle_cores(void) { return resolve_threads(0); }

/* ------------------------------------------------------------------------
 * Philox4x32-10 (Salmon et al., SC 2011).  One round maps counter (c0..c3)
 * and key (k0, k1) to
 *     (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0))
 * with M0 = 0xD2511F53, M1 = 0xCD9E8D57; after each round the key grows by
 * the Weyl increments (0x9E3779B9, 0xBB67AE85).  Ten rounds.
 * ------------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    const int rounds = g_mutation == MUT_PHILOX_9_ROUNDS ? 9 : 10;
    for (int r = 0; r < rounds; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        const uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* The uniform of token v in a row with counter offset `off` under `seed`:
 * Philox word (v & 3) of counter (v >> 2, lo(off), hi(off), 0x53414D50),
 * key (lo(seed), hi(seed)); u = ((w >> 9) + 0.5) * 2^-23, exactly
 * representable in fp32 and strictly inside (0, 1). */
double oracle_sample_uniform(uint64_t seed, int64_t off, int32_t v)
{
    const uint32_t ctr[4] = {(uint32_t)v >> 2, (uint32_t)(uint64_t)off, (uint32_t)((uint64_t)off >> 32),
                             0x53414D50u};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    return ((double)(w[v & 3] >> 9) + 0.5) * ldexp(1.0, -23);
}

/* Gumbel-max sampling over z (f64 [rows x V], row stride V).
 *   temperature  [rows] or NULL (= 1); T <= 0 selects argmax z (greedy)
 *   mask         [rows x mask_words] or NULL: token v is allowed when bit
 *                (v % 32) of word v / 32 is set
 *   offsets      [rows] or NULL (= the row index): the counter offset
 * out_ids[i] = the allowed token with the largest score z/T + g (greedy: z),
 * ties to the smaller id; -1 when no token is allowed.  out_score[i] is
 * that score, out_second[i] the largest score of any other allowed token
 * (-inf if none), for near-tie checks. */
int oracle_sample(const double* z, int32_t rows, int32_t V, const float* temperature, const uint32_t* mask,
                  int32_t mask_words, uint64_t seed, const int64_t* offsets, int32_t* out_ids,
                  double* out_score, double* out_second)
{
    if (!z || rows < 0 || V <= 0 || !out_ids || !out_score || !out_second) return ORACLE_ERR_ARG;
    if (mask && mask_words < (V + 31) / 32) return ORACLE_ERR_ARG;
    for (int32_t i = 0; i < rows; ++i) {
        const double T = temperature ? (double)temperature[i] : 1.0;
        const int greedy = T <= 0.0;
        const int64_t off = offsets ? offsets[i] : (int64_t)i;
        int32_t best = -1;
        double bs = -INFINITY, second = -INFINITY;
        for (int32_t v = 0; v < V; ++v) {
            if (mask && g_mutation != MUT_MASK_IGNORED &&
                !((mask[(int64_t)i * mask_words + v / 32] >> (v % 32)) & 1u))
                continue;
            const double x = z[(int64_t)i * V + v];
            double s;
            if (greedy) {
                s = x;
            } else {
                const double u = oracle_sample_uniform(seed, off, v);
                double g = -log(-log(u));
                if (g_mutation == MUT_GUMBEL_SIGN) g = -g;
                s = (g_mutation == MUT_TEMP_TIMES ? x * T : x / T) + g;
            }
            if (best < 0 || s > bs) {
                if (best >= 0) second = bs;
                best = v;
                bs = s;
            } else if (s > second) {
                second = s;
            }
        }
        out_ids[i] = best;
        out_score[i] = best >= 0 ? bs : -INFINITY;
        out_second[i] = second;
    }
    return ORACLE_OK;
}
