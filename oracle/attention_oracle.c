/*
 * attention_oracle.c -- plain, slow, fp64 CPU reference for the attention
 * forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; it is used by the tests, by the smoke check and by the
 * benchmark's CPU-baseline leg.  It shares no code, header or constant with
 * the CUDA path.
 *
 * What it computes (the plain definition, no blocking, no online softmax):
 *
 *   For every packed sequence b, query row i in [0, Lq_b) and head h:
 *     off      = Lk_b - Lq_b                     (bottom-right alignment)
 *     V(i)     = { j in [0, Lk_b) :
 *                    (!causal || j <= i + off)
 *                 && (wl < 0  || j >= i + off - wl)
 *                 && (wr < 0  || j <= i + off + wr) }
 *     s_ij     = scale * sum_c q[i,c] * k[j,c]              (fp64)
 *     m        = max_{j in V(i)} s_ij
 *     L        = m + ln( sum_{j in V(i)} exp(s_ij - m) )    (natural log)
 *     O[i,:]   = sum_{j in V(i)} exp(s_ij - L) * v[j,:]
 *     V(i) empty  ->  O = 0, L = -inf.
 *
 * Sources:
 *   - packed sequences given by cu_seqlens_q / cu_seqlens_k, softmax_scale,
 *     causal, window_size and return_softmax_lse:  vLLM API page
 *     "vllm.v1.attention.backends.mla.prefill.flash_attn", FA4MLAPrefillKernel
 *     (CompileKey fields) and FlashAttnPrefillBackend (run_prefill_new_tokens
 *     is causal with cu_seqlens_q == cu_seqlens_k; run_prefill_context_chunk is
 *     non-causal and returns the LSE).
 *   - "sliding-window prefill is always causal": same page,
 *     FA4MLAPrefillKernel._is_valid_warmup_shape_probe.
 *   - chunked prefill with q shorter than k is a tested configuration: sglang
 *     PR #41344 (FA4 path on Blackwell), "Accuracy Tests".  The bottom-right
 *     alignment of the causal diagonal for Lq < Lk is the reading taken here.
 *   - the LSE is stored head-major, [H, total_q]: FA4SplitKVCombineKernel on
 *     the flash_attn page (the LSE buffer is allocated [num_heads, total_q]
 *     and transposed).
 *   - sparse-MLA decode (one query row per token, rows gathered by per-token
 *     indices, head size 576 = 512 latent + 64 rope, V = the 512 latent
 *     columns, BF16 cache only): vLLM API page
 *     "vllm.v1.attention.backends.mla.flashattn_mla_sparse",
 *     FlashAttnMLASparseFA4Backend and _fa4_varlen_scalars.
 *
 * Inputs are bf16 bit patterns (uint16_t); each is widened exactly to double.
 * Every result is fp64.  The window bounds are inclusive; -1 means unbounded.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes of this file (its own; the product library has its own). */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEMORY 2

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The valid-key predicate of the definition above. */
static int key_is_valid(int64_t i, int64_t j, int64_t lq, int64_t lk,
                        int causal, int64_t wl, int64_t wr)
{
    int64_t off = lk - lq;
    if (j < 0 || j >= lk) return 0;
    if (causal && j > i + off) return 0;
    if (wl >= 0 && j < i + off - wl) return 0;
    if (wr >= 0 && j > i + off + wr) return 0;
    return 1;
}

/*
 * Attention of one query vector over an explicit list of key/value rows.
 * q: d_qk doubles.  krows[n]/vrows[n]: bf16 rows (d_qk and d_v wide).
 * scores: scratch of n doubles.  out: d_v doubles.  *lse: natural-log LSE.
 * Two plain passes over the scores: the maximum, then the sum.
 */
static void attend_rows(const double *q, int d_qk, int d_v, double scale,
                        const uint16_t *const *krows,
                        const uint16_t *const *vrows, int64_t n,
                        double *scores, double *out, double *lse)
{
    for (int c = 0; c < d_v; ++c) out[c] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d_qk; ++c)
            dot += q[c] * bf16_bits_to_double(krows[j][c]);
        scores[j] = scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) sum += exp(scores[j] - m);
    double L = m + log(sum);
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(scores[j] - L);
        for (int c = 0; c < d_v; ++c)
            out[c] += p * bf16_bits_to_double(vrows[j][c]);
    }
    *lse = L;
}

/* Sequence that packed token t belongs to (cu is non-decreasing). */
static int find_sequence(const int32_t *cu, int batch, int64_t t)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    /* Skip empty sequences that share this start offset. */
    while (lo + 1 < batch && (int64_t)cu[lo + 1] <= t) ++lo;
    return lo;
}

/*
 * Varlen attention forward.
 *   q [total_q, H, d_qk], k [total_k, H_k, d_qk], v [total_k, H_k, d_v]: bf16.
 *   Query head h reads key/value head h / (H / H_k).
 *   Rows are (token, head) pairs flattened as token * H + head.  With
 *   row_ids == NULL all total_q * H rows are computed, in that order; else the
 *   num_rows listed rows.  out: [rows, d_v] doubles; lse: [rows] doubles.
 *   num_threads <= 0 leaves the OpenMP default.
 */
int oracle_varlen_attention(const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, const int32_t *cu_seqlens_q,
                            const int32_t *cu_seqlens_k, int batch,
                            int num_heads, int num_heads_k, int d_qk, int d_v,
                            double softmax_scale, int causal, int window_left,
                            int window_right, int64_t num_rows,
                            const int64_t *row_ids, double *out, double *lse,
                            int num_threads)
{
    if (!q || !cu_seqlens_q || !cu_seqlens_k || !out || !lse)
        return ORACLE_BAD_ARG;
    if (batch < 1 || num_heads < 1 || num_heads_k < 1 ||
        num_heads % num_heads_k != 0 || d_qk < 1 || d_v < 1)
        return ORACLE_BAD_ARG;
    int64_t total_q = cu_seqlens_q[batch];
    if (row_ids == NULL) num_rows = total_q * num_heads;
    int group = num_heads / num_heads_k;
    int64_t max_lk = 0;
    for (int b = 0; b < batch; ++b) {
        int64_t lk = (int64_t)cu_seqlens_k[b + 1] - cu_seqlens_k[b];
        int64_t lq = (int64_t)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
        if (lk < 0 || lq < 0) return ORACLE_BAD_ARG;
        if (lk > max_lk) max_lk = lk;
    }
    if (max_lk > 0 && (!k || !v)) return ORACLE_BAD_ARG;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *qd = (double *)malloc(sizeof(double) * (size_t)d_qk);
        double *scores = (double *)malloc(sizeof(double) * (size_t)(max_lk + 1));
        const uint16_t **krows =
            (const uint16_t **)malloc(sizeof(void *) * (size_t)(max_lk + 1));
        const uint16_t **vrows =
            (const uint16_t **)malloc(sizeof(void *) * (size_t)(max_lk + 1));
        if (!qd || !scores || !krows || !vrows) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < num_rows; ++r) {
                int64_t flat = row_ids ? row_ids[r] : r;
                int64_t t = flat / num_heads;
                int h = (int)(flat % num_heads);
                int hk = h / group;
                int b = find_sequence(cu_seqlens_q, batch, t);
                int64_t lq = (int64_t)cu_seqlens_q[b + 1] - cu_seqlens_q[b];
                int64_t lk = (int64_t)cu_seqlens_k[b + 1] - cu_seqlens_k[b];
                int64_t i = t - cu_seqlens_q[b];
                for (int c = 0; c < d_qk; ++c)
                    qd[c] = bf16_bits_to_double(
                        q[((size_t)t * num_heads + h) * d_qk + c]);
                int64_t n = 0;
                for (int64_t j = 0; j < lk; ++j) {
                    if (!key_is_valid(i, j, lq, lk, causal, window_left,
                                      window_right))
                        continue;
                    int64_t kt = cu_seqlens_k[b] + j;
                    krows[n] = k + ((size_t)kt * num_heads_k + hk) * d_qk;
                    vrows[n] = v + ((size_t)kt * num_heads_k + hk) * d_v;
                    ++n;
                }
                attend_rows(qd, d_qk, d_v, softmax_scale, krows, vrows, n,
                            scores, out + (size_t)r * d_v, lse + r);
            }
        }
        free(qd);
        free(scores);
        free((void *)krows);
        free((void *)vrows);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Sparse-MLA decode: one query row per token, all heads share the gathered
 * latent rows (multi-query form).
 *   q [T, H, 576] bf16; kv_cache [num_pages, page_size, 576] bf16.
 *   page_table [T, max_pages_per_tok] int32: physical page of each logical
 *   page of the token's context.  topk_idx [T, topk] int32: logical positions
 *   in the token's context.  Logical position p lives in physical row
 *   page_table[t, p / page_size] * page_size + p % page_size.
 *   Scores use all 576 columns; the value is the first 512 columns.
 *   A slot whose position is negative or past the context, or whose page id is
 *   outside [0, num_pages), contributes nothing.
 *   Rows are flattened as token * H + head; out [rows, 512], lse [rows].
 */
int oracle_sparse_mla_decode(const uint16_t *q, const uint16_t *kv_cache,
                             const int32_t *page_table,
                             const int32_t *topk_idx, int num_tokens,
                             int num_heads, int topk, int num_pages,
                             int max_pages_per_tok, int page_size,
                             double softmax_scale, int64_t num_rows,
                             const int64_t *row_ids, double *out, double *lse,
                             int num_threads)
{
    const int d_qk = 576, d_v = 512;
    if (!q || !kv_cache || !page_table || !topk_idx || !out || !lse)
        return ORACLE_BAD_ARG;
    if (num_tokens < 0 || num_heads < 1 || topk < 0 || num_pages < 0 ||
        max_pages_per_tok < 0 || page_size < 1)
        return ORACLE_BAD_ARG;
    if (row_ids == NULL) num_rows = (int64_t)num_tokens * num_heads;
    int64_t context = (int64_t)max_pages_per_tok * page_size;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *qd = (double *)malloc(sizeof(double) * d_qk);
        double *scores = (double *)malloc(sizeof(double) * (size_t)(topk + 1));
        const uint16_t **rows =
            (const uint16_t **)malloc(sizeof(void *) * (size_t)(topk + 1));
        if (!qd || !scores || !rows) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < num_rows; ++r) {
                int64_t flat = row_ids ? row_ids[r] : r;
                int64_t t = flat / num_heads;
                int h = (int)(flat % num_heads);
                for (int c = 0; c < d_qk; ++c)
                    qd[c] = bf16_bits_to_double(
                        q[((size_t)t * num_heads + h) * d_qk + c]);
                int64_t n = 0;
                for (int s = 0; s < topk; ++s) {
                    int64_t p = topk_idx[(size_t)t * topk + s];
                    if (p < 0 || p >= context) continue;
                    int64_t page =
                        page_table[(size_t)t * max_pages_per_tok + p / page_size];
                    if (page < 0 || page >= num_pages) continue;
                    int64_t phys = page * page_size + p % page_size;
                    rows[n++] = kv_cache + (size_t)phys * d_qk;
                }
                /* K and V are the same gathered rows: V is their prefix. */
                attend_rows(qd, d_qk, d_v, softmax_scale, rows, rows, n,
                            scores, out + (size_t)r * d_v, lse + r);
            }
        }
        free(qd);
        free(scores);
        free((void *)rows);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Merge of two partial attention results of the same query rows over
 * disjoint key sets A and B, weighted by their log-sum-exps:
 *   L = ln(e^{L_A} + e^{L_B}),   O = e^{L_A - L} O_A + e^{L_B - L} O_B.
 * An LSE of -inf marks an empty part (weight 0); both empty gives O = 0 and
 * L = -inf.  Source: merge_attn_states on the vLLM page
 * "vllm.v1.attention.backends.mla.prefill.flash_attn" (the context-chunk
 * partial, non-causal with LSE, and the new-token partial, causal, are merged
 * by their LSEs; FlashAttnPrefillBackend).
 *   o_a, o_b: [rows, d]; lse_a, lse_b: [rows]; out: [rows, d]; lse: [rows].
 */
int oracle_merge_states(const double *o_a, const double *lse_a,
                        const double *o_b, const double *lse_b, int64_t rows,
                        int d, double *out, double *lse)
{
    if (!o_a || !lse_a || !o_b || !lse_b || !out || !lse || rows < 0 || d < 1)
        return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < rows; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        double m = la > lb ? la : lb;
        if (m == -INFINITY) {
            for (int c = 0; c < d; ++c) out[(size_t)r * d + c] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double L = m + log(exp(la - m) + exp(lb - m));
        double wa = exp(la - L), wb = exp(lb - L);
        for (int c = 0; c < d; ++c)
            out[(size_t)r * d + c] =
                wa * o_a[(size_t)r * d + c] + wb * o_b[(size_t)r * d + c];
        lse[r] = L;
    }
    return ORACLE_OK;
}

/* Number of OpenMP threads a parallel region would use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
