/*
 * Scaled dot-product attention: fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against.  It shares no code,
 * header, table or constant with the CUDA path; only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * What it computes, per (batch b, head h, query row i):
 *
 *   out[i] = sum_j softmax_j( scale * q_i . k_j + M_ij ) v_j
 *
 * with M_ij = 0 for an allowed (query, key) pair and -inf for a forbidden
 * one, applied before the softmax.  Sources:
 *   - "Attention from First Principles", section 1 ("In one line") and
 *     section 4 "Tiny example" (score, scale, causal mask, row softmax,
 *     multiply by V, worked by hand);
 *   - "Attention from Scratch" (kube-dojo), Part 2 "Scaled Dot-Product
 *     Attention by Hand" (general T_q x T_k form, d_v may differ from d_k,
 *     softmax over the key axis) and Part 3 "Masks, Causality, and Padding"
 *     (causal allowed-mask j <= i, key-padding mask over key columns, the two
 *     combined with logical AND);
 *   - "Self-Attention", sections "Scaled Dot-Product Attention" and "Causal
 *     Masking" (additive mask M_ij = 0 for j <= i, -inf otherwise);
 *   - "Scaled dot-product attention with masking", "The math" and "Adding the
 *     causal mask" (decode: a single query sees every cached key).
 *
 * Readings where the pages leave a step open:
 *   1. Forbidden keys are EXCLUDED from the max, the sum and the mixture.
 *      This is the exact value of adding -inf before the softmax, written
 *      without inf arithmetic.
 *   2. Causal with T_q != T_k aligns the last query with the last key:
 *      key j is visible from query i iff j <= i + (T_k - T_q).  For T_q ==
 *      T_k this is the pages' lower-triangular mask; for T_q == 1 it is the
 *      pages' decode rule (the new query sees the whole cache).
 *   3. Key padding is right padding: with per-sequence length L_b, keys
 *      j >= L_b are masked.
 *   4. A query row that can see no key, and (when query_padding is set) a
 *      padded query row i >= L_b, output exact zeros.  The pages raise an
 *      error for an all-masked row ("Attention from Scratch", Part 2 and the
 *      "Common Mistakes" table); an error cannot be raised from inside a
 *      batched kernel, so the library defines the row as zero.
 *   5. Softmax is max-subtracted before exponentiation ("Attention from
 *      Scratch", Part 7, stable-softmax habit).
 *
 * Inputs are read as float32 or as bfloat16 bit patterns and widened exactly
 * to double; every sum is a double sum in index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1

/* Exact widening of one stored element to double. */
static double load_elem(const void *base, int dtype, size_t idx)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[idx];
    /* bfloat16 is the top half of an IEEE float32: shift the 16 stored bits up. */
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Is key j visible from query i?  (readings 2 and 3 above)  `off` is the
 * absolute position of query 0 among the keys: Skv - Sq when the last query
 * is aligned with the last key, L_b - Sq for a chunk of queries at the end of
 * a cached sequence of L_b positions.
 */
static int key_visible(int i, int j, int off, int causal, int Lb)
{
    if (j >= Lb)
        return 0;
    if (causal && j > i + off)
        return 0;
    return 1;
}

/*
 * One output row.  q_bh, k_bh, v_bh are element offsets of the (b, h) slices.
 * s_row is caller scratch of length Skv.  w_row, if not NULL, receives the
 * attention weights of this row (zero for forbidden keys).
 */
static void attention_row(const void *q, const void *k, const void *v, int dtype,
                          size_t q_bh, size_t k_bh, size_t v_bh, int i, int off, int Skv,
                          int Dk, int Dv, double scale, int causal, int Lb, int query_padding,
                          double *out_row, double *w_row, double *s_row, double *lse)
{
    int d, j;
    for (d = 0; d < Dv; d++)
        out_row[d] = 0.0;
    if (w_row)
        for (j = 0; j < Skv; j++)
            w_row[j] = 0.0;

    if (lse)
        *lse = -INFINITY;
    /* reading 4: a padded query row is zero */
    if (query_padding && i >= Lb)
        return;

    /* scores of the visible keys, and their maximum */
    int any = 0;
    double m = 0.0;
    for (j = 0; j < Skv; j++) {
        if (!key_visible(i, j, off, causal, Lb))
            continue;
        double dot = 0.0;
        for (d = 0; d < Dk; d++)
            dot += load_elem(q, dtype, q_bh + (size_t)i * Dk + d) *
                   load_elem(k, dtype, k_bh + (size_t)j * Dk + d);
        s_row[j] = scale * dot;
        if (!any || s_row[j] > m)
            m = s_row[j];
        any = 1;
    }
    /* reading 4: a row that sees no key is zero */
    if (!any)
        return;

    /* max-subtracted softmax over the key axis, then the mixture of V rows */
    double z = 0.0;
    for (j = 0; j < Skv; j++)
        if (key_visible(i, j, off, causal, Lb))
            z += exp(s_row[j] - m);
    /* log-sum-exp of the visible scores: log(sum_j exp(s_j)) = m + log(z) */
    if (lse)
        *lse = m + log(z);
    for (j = 0; j < Skv; j++) {
        if (!key_visible(i, j, off, causal, Lb))
            continue;
        double w = exp(s_row[j] - m) / z;
        if (w_row)
            w_row[j] = w;
        for (d = 0; d < Dv; d++)
            out_row[d] += w * load_elem(v, dtype, v_bh + (size_t)j * Dv + d);
    }
}

static int sequence_length(const int32_t *kv_len, int b, int Skv)
{
    if (!kv_len)
        return Skv;
    int L = kv_len[b];
    if (L < 0)
        L = 0;
    if (L > Skv)
        L = Skv;
    return L;
}

static int check_dims(int B, int H, int Sq, int Skv, int Dk, int Dv, int dtype)
{
    if (B < 0 || H < 0 || Sq < 0 || Skv < 0 || Dk <= 0 || Dv <= 0)
        return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16)
        return -1;
    return 0;
}

/*
 * Grouped-query attention ("Attention from First Principles", section 5 "The
 * full multi-head computation" and "MHA, GQA, MQA -- the KV cache lever";
 * "Scaled dot-product attention with masking", "Grouped-query attention
 * (GQA)"): q has H heads, k and v have Hkv heads, Hkv divides H, and query head
 * h attends with key/value head h / (H / Hkv) -- the head the pages'
 * repeat_interleave(H / Hkv) of K and V places at position h.  Hkv == H is
 * ordinary multi-head attention, Hkv == 1 is multi-query attention.
 *
 * q: (B,H,Sq,Dk)  k: (B,Hkv,Skv,Dk)  v: (B,Hkv,Skv,Dv)
 * out: (B,H,Sq,Dv) doubles.  weights: (B,H,Sq,Skv) doubles or NULL.
 * kv_len: host int32[B] or NULL (all keys valid).  query_padding: 1 makes
 * query rows i >= L_b zero (self-attention prefill over right-padded
 * batches), 0 leaves them as computed (decode, cross-attention).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_attention_gqa(const void *q, const void *k, const void *v, int dtype, double *out,
                         double *weights, int B, int H, int Hkv, int Sq, int Skv, int Dk, int Dv,
                         double scale, int causal, const int32_t *kv_len, int query_padding,
                         int nthreads)
{
    if (check_dims(B, H, Sq, Skv, Dk, Dv, dtype) || !out || Hkv <= 0 || H % Hkv)
        return -1;
    const int G = H / Hkv;
    long long n_bh = (long long)B * H;
    long long p;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads > 0 ? nthreads : 1)
    for (p = 0; p < n_bh; p++) {
        int b = (int)(p / H), h = (int)(p % H);
        size_t pkv = (size_t)b * Hkv + h / G; /* the key/value head of query head h */
        int Lb = sequence_length(kv_len, b, Skv);
        double *s_row = (double *)malloc(sizeof(double) * (Skv > 0 ? Skv : 1));
        for (int i = 0; i < Sq; i++) {
            double *w_row = weights ? weights + ((size_t)p * Sq + i) * Skv : NULL;
            attention_row(q, k, v, dtype, (size_t)p * Sq * Dk, pkv * Skv * Dk, pkv * Skv * Dv, i,
                          Skv - Sq, Skv, Dk, Dv, scale, causal, Lb, query_padding,
                          out + ((size_t)p * Sq + i) * Dv, w_row, s_row, NULL);
        }
        free(s_row);
    }
    return 0;
}

/* Multi-head attention: the grouped form with one key/value head per query head. */
int oracle_attention(const void *q, const void *k, const void *v, int dtype, double *out,
                     double *weights, int B, int H, int Sq, int Skv, int Dk, int Dv,
                     double scale, int causal, const int32_t *kv_len, int query_padding,
                     int nthreads)
{
    return oracle_attention_gqa(q, k, v, dtype, out, weights, B, H, H, Sq, Skv, Dk, Dv, scale,
                                causal, kv_len, query_padding, nthreads);
}

/*
 * The same definition evaluated only at chosen rows.  rows holds n_rows
 * triples (b, h, i); out receives n_rows x Dv doubles in that order.  Used to
 * check outputs at full benchmark sizes one row at a time.
 */
int oracle_attention_rows_gqa(const void *q, const void *k, const void *v, int dtype, double *out,
                              int B, int H, int Hkv, int Sq, int Skv, int Dk, int Dv, double scale,
                              int causal, const int32_t *kv_len, int query_padding,
                              const int64_t *rows, long long n_rows, int nthreads)
{
    if (check_dims(B, H, Sq, Skv, Dk, Dv, dtype) || !out || (n_rows > 0 && !rows) || Hkv <= 0 ||
        H % Hkv)
        return -1;
    for (long long r = 0; r < n_rows; r++) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Sq)
            return -1;
    }
    const int G = H / Hkv;
    long long r;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads > 0 ? nthreads : 1)
    for (r = 0; r < n_rows; r++) {
        int b = (int)rows[3 * r], h = (int)rows[3 * r + 1], i = (int)rows[3 * r + 2];
        size_t p = (size_t)b * H + h;
        size_t pkv = (size_t)b * Hkv + h / G;
        int Lb = sequence_length(kv_len, b, Skv);
        double *s_row = (double *)malloc(sizeof(double) * (Skv > 0 ? Skv : 1));
        attention_row(q, k, v, dtype, p * Sq * Dk, pkv * Skv * Dk, pkv * Skv * Dv, i, Skv - Sq, Skv,
                      Dk, Dv, scale, causal, Lb, query_padding, out + (size_t)r * Dv, NULL, s_row,
                      NULL);
        free(s_row);
    }
    return 0;
}

int oracle_attention_rows(const void *q, const void *k, const void *v, int dtype, double *out,
                          int B, int H, int Sq, int Skv, int Dk, int Dv, double scale, int causal,
                          const int32_t *kv_len, int query_padding, const int64_t *rows,
                          long long n_rows, int nthreads)
{
    return oracle_attention_rows_gqa(q, k, v, dtype, out, B, H, H, Sq, Skv, Dk, Dv, scale, causal,
                                     kv_len, query_padding, rows, n_rows, nthreads);
}

/*
 * Prefill of a chunk of Sq new queries against a KV cache, with the
 * log-sum-exp of every row.  Sequence b holds L_b = cache_len[b] valid cache
 * positions, the last Sq of which are the chunk's own keys (the cache append
 * of "Scaled dot-product attention with masking", "The full multi-head
 * computation"); query i sits at absolute position L_b - Sq + i and sees the
 * keys j <= L_b - Sq + i ("Attention from scratch" (open-llm-engineering),
 * "KV cache position drift": cache positions and token positions must agree).
 * A query with a negative position (L_b < Sq: the chunk is longer than the
 * sequence) sees no key: its row is zero.
 *
 * q: (B,H,Sq,Dk)  k: (B,Hkv,Skv,Dk)  v: (B,Hkv,Skv,Dv)  out: (B,H,Sq,Dv) doubles.
 * lse: (B,H,Sq) doubles or NULL: log(sum_j exp(scale * q_i.k_j)) over the
 * visible keys, -inf for a row that sees none.  cache_len: host int32[B] or
 * NULL (every L_b = Skv).  Returns 0, or -1 on a bad argument.
 */
int oracle_attention_cache(const void *q, const void *k, const void *v, int dtype, double *out,
                           double *lse, int B, int H, int Hkv, int Sq, int Skv, int Dk, int Dv,
                           double scale, const int32_t *cache_len, int nthreads)
{
    if (check_dims(B, H, Sq, Skv, Dk, Dv, dtype) || !out || Hkv <= 0 || H % Hkv)
        return -1;
    const int G = H / Hkv;
    long long n_bh = (long long)B * H;
    long long p;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads > 0 ? nthreads : 1)
    for (p = 0; p < n_bh; p++) {
        int b = (int)(p / H), h = (int)(p % H);
        size_t pkv = (size_t)b * Hkv + h / G;
        int Lb = sequence_length(cache_len, b, Skv);
        double *s_row = (double *)malloc(sizeof(double) * (Skv > 0 ? Skv : 1));
        for (int i = 0; i < Sq; i++)
            attention_row(q, k, v, dtype, (size_t)p * Sq * Dk, pkv * Skv * Dk, pkv * Skv * Dv, i,
                          Lb - Sq, Skv, Dk, Dv, scale, 1, Lb, 0, out + ((size_t)p * Sq + i) * Dv,
                          NULL, s_row, lse ? lse + (size_t)p * Sq + i : NULL);
        free(s_row);
    }
    return 0;
}
