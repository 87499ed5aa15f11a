/*
 * CPU oracle for speculative-decoding verify attention.  TEST INFRASTRUCTURE
 * ONLY: the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg call this file; the product path never does.  It shares no code, header
 * or constant with the CUDA library.
 *
 * What it computes (plain definition, fp64 throughout, no blocking, no
 * splitting, no online softmax):
 *
 *   The verify step of speculative decoding scores a block of T drafted
 *   tokens in one forward pass.  Source: "I pushed Qwen3.8-27B to 124 tps on
 *   a single request on a RTX 3090", bullet "Split-KV attention kernel for
 *   the verify step" (attention of a few verify queries against a long KV
 *   cache; the split-KV kernel is an exact reorganisation of that attention,
 *   and "speculative decoding is exact by construction", closing paragraph
 *   of the same page).  The T verify tokens' own K/V are already in the
 *   paged cache, so sequence b holds L_b keys and verify token t sees keys
 *   j <= L_b - T + t (bottom-right causal mask).
 *
 *   The cache is paged (16-token pages, block table per sequence) and stored
 *   as bf16, fp8-e4m3 or int8 with one fp32 scale per (token, kv-head):
 *   "I pushed Qwen3.8-27B to 381 tps for a single request on a RTX 3090",
 *   "What we had" (fp8 KV cache) and "DFlash2 past 64k" (int8 cache, vLLM
 *   16-token blocks).  The same page's "KVarN 4/2-bit KV cache" bullet adds
 *   4-bit and 2-bit caches without describing their format; the reading
 *   used here is the int8 format with fewer bits: signed two's-complement
 *   codes (int4 in [-8, 7], int2 in [-2, 1]; the encoder uses +-7 / +-1)
 *   times the same per-(token, kv-head) fp32 scale, packed little-end first
 *   (element d of a row sits in bits (d * bits) % 8 .. of byte d * bits / 8).
 *
 *   For sequence b, verify token t, query head h, kv head g = h / G:
 *     Khat[j] = decode(k_pages[page(j), j % 16, g, :]) * k_scale[page, slot, g]
 *     s_j     = (1/sqrt(D)) * sum_d q[b,t,h,d] * Khat[j,d]      for j <= p_t
 *     m       = max_j s_j,  Z = sum_j exp(s_j - m),  lse = m + ln Z
 *     out     = sum_j exp(s_j - lse) * Vhat[j, :]
 *   (bf16 caches carry no scale: the scale is 1.)
 *
 * Layouts (row-major, contiguous):
 *   q           uint16 (bf16 bits) [B, T, Hq, D]
 *   k/v_pages   [num_pages, 16, Hkv, D] of bf16 bits / e4m3 bytes / int8;
 *               int4 / int2: [num_pages, 16, Hkv, D * bits / 8] packed bytes
 *   k/v_scale   float [num_pages, 16, Hkv]       (ignored for bf16)
 *   block_table int32 [B, bt_stride]
 *   seq_lens    int32 [B]   (includes the T verify tokens)
 *   out         double [B, T, Hq, D],  lse double [B, T, Hq]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_PAGE 16

enum { ORACLE_BF16 = 0, ORACLE_E4M3 = 1, ORACLE_INT8 = 2, ORACLE_INT4 = 3, ORACLE_INT2 = 4 };

/* bf16 is the top half of an IEEE-754 binary32. */
double oracle_decode_bf16(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * (2^-6 * m/8); S.1111.111 is NaN; there are no infinities (max 448). */
double oracle_decode_e4m3(uint8_t bits)
{
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

double oracle_decode_int8(int8_t v) { return (double)v; }

/* Element idx of a packed array of `bits`-bit two's-complement codes
 * (bits = 4 or 2): the field at bit (idx * bits) % 8 of byte idx * bits / 8,
 * sign-extended. */
double oracle_decode_packed(const uint8_t *base, size_t idx, int bits)
{
    size_t bit = idx * (size_t)bits;
    int field = (base[bit / 8] >> (bit % 8)) & ((1 << bits) - 1);
    if (field >= (1 << (bits - 1)))
        field -= 1 << bits;
    return (double)field;
}

static double decode_elem(const void *base, size_t idx, int dtype)
{
    switch (dtype) {
    case ORACLE_BF16: return oracle_decode_bf16(((const uint16_t *)base)[idx]);
    case ORACLE_E4M3: return oracle_decode_e4m3(((const uint8_t *)base)[idx]);
    case ORACLE_INT4: return oracle_decode_packed((const uint8_t *)base, idx, 4);
    case ORACLE_INT2: return oracle_decode_packed((const uint8_t *)base, idx, 2);
    default: return oracle_decode_int8(((const int8_t *)base)[idx]);
    }
}

typedef struct {
    const uint16_t *q;
    const void *k_pages, *v_pages;
    const float *k_scale, *v_scale;
    const int32_t *block_table;
    int bt_stride;
    const int32_t *seq_lens;
    int num_seqs, T, Hq, Hkv, D, dtype;
} problem;

/* Dequantised row of the cache: token j of sequence b, kv head g. */
static void dequant_row(const problem *P, const void *pages, const float *scale,
                        int b, int j, int g, double *dst)
{
    int page = P->block_table[(size_t)b * P->bt_stride + j / ORACLE_PAGE];
    int slot = j % ORACLE_PAGE;
    size_t row = ((size_t)page * ORACLE_PAGE + slot) * P->Hkv + g;
    double s = 1.0;
    if (P->dtype != ORACLE_BF16)
        s = (double)scale[row];
    for (int d = 0; d < P->D; ++d)
        dst[d] = decode_elem(pages, row * P->D + d, P->dtype) * s;
}

/* Attention of one (b, t, h) query over the visible keys that fall in
 * [key_begin, key_end).  With [0, L_b) this is the whole definition above.
 * An empty visible range gives lse = -inf and out = 0 (nothing attended).
 * Returns 0, or -1 on allocation failure. */
static int attend_one(const problem *P, int b, int t, int h, int key_begin,
                      int key_end, double *out, double *lse)
{
    const int D = P->D;
    const int G = P->Hq / P->Hkv;
    const int g = h / G;
    const int L = P->seq_lens[b];
    const int last_visible = L - P->T + t; /* bottom-right causal mask */
    int hi = key_end < last_visible + 1 ? key_end : last_visible + 1;
    int lo = key_begin > 0 ? key_begin : 0;
    const uint16_t *qrow = P->q + (((size_t)b * P->T + t) * P->Hq + h) * D;

    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (hi <= lo) {
        *lse = -INFINITY;
        return 0;
    }
    int n = hi - lo;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    if (!s || !qd || !row) {
        free(s); free(qd); free(row);
        return -1;
    }
    for (int d = 0; d < D; ++d)
        qd[d] = oracle_decode_bf16(qrow[d]);
    const double scale = 1.0 / sqrt((double)D);

    /* scores */
    for (int j = lo; j < hi; ++j) {
        dequant_row(P, P->k_pages, P->k_scale, b, j, g, row);
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += qd[d] * row[d];
        s[j - lo] = scale * acc;
    }
    /* explicit softmax */
    double m = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (s[i] > m) m = s[i];
    double Z = 0.0;
    for (int i = 0; i < n; ++i)
        Z += exp(s[i] - m);
    const double l = m + log(Z);
    for (int j = lo; j < hi; ++j) {
        const double p = exp(s[j - lo] - l);
        dequant_row(P, P->v_pages, P->v_scale, b, j, g, row);
        for (int d = 0; d < D; ++d)
            out[d] += p * row[d];
    }
    *lse = l;
    free(s); free(qd); free(row);
    return 0;
}

static int check_problem(const problem *P)
{
    if (!P->q || !P->k_pages || !P->v_pages || !P->block_table || !P->seq_lens)
        return -1;
    if (P->num_seqs < 0 || P->T < 1 || P->Hq < 1 || P->Hkv < 1 || P->D < 1)
        return -1;
    if (P->Hq % P->Hkv != 0)
        return -1;
    if (P->dtype < ORACLE_BF16 || P->dtype > ORACLE_INT2)
        return -1;
    if (P->dtype == ORACLE_INT2 && P->D % 4 != 0)
        return -1;
    if (P->dtype == ORACLE_INT4 && P->D % 2 != 0)
        return -1;
    if (P->dtype != ORACLE_BF16 && (!P->k_scale || !P->v_scale))
        return -1;
    for (int b = 0; b < P->num_seqs; ++b) {
        if (P->seq_lens[b] < P->T)
            return -1;
        if ((P->seq_lens[b] + ORACLE_PAGE - 1) / ORACLE_PAGE > P->bt_stride)
            return -1;
    }
    return 0;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Number of threads the parallel loops will use. */
int oracle_max_threads(int nthreads)
{
#ifdef _OPENMP
    set_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Full verify attention: every (b, t, h).  Returns 0 on success. */
int oracle_verify_attn(const uint16_t *q, const void *k_pages, const void *v_pages,
                       const float *k_scale, const float *v_scale,
                       const int32_t *block_table, int bt_stride,
                       const int32_t *seq_lens, int num_seqs, int T, int Hq,
                       int Hkv, int D, int kv_dtype, double *out, double *lse,
                       int nthreads)
{
    problem P = {q, k_pages, v_pages, k_scale, v_scale, block_table, bt_stride,
                 seq_lens, num_seqs, T, Hq, Hkv, D, kv_dtype};
    if (check_problem(&P) || !out || !lse)
        return -1;
    set_threads(nthreads);
    const long total = (long)num_seqs * T * Hq;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (long i = 0; i < total; ++i) {
        int h = (int)(i % Hq);
        int t = (int)((i / Hq) % T);
        int b = (int)(i / ((long)Hq * T));
        failed |= attend_one(&P, b, t, h, 0, seq_lens[b], out + (size_t)i * D,
                             lse + i) != 0;
    }
    return failed ? -1 : 0;
}

/* Selected outputs only: rows[3*i .. 3*i+2] = (b, t, h).  out is [n_rows, D]. */
int oracle_verify_attn_rows(const uint16_t *q, const void *k_pages, const void *v_pages,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_table, int bt_stride,
                            const int32_t *seq_lens, int num_seqs, int T, int Hq,
                            int Hkv, int D, int kv_dtype, const int32_t *rows,
                            int n_rows, double *out, double *lse, int nthreads)
{
    problem P = {q, k_pages, v_pages, k_scale, v_scale, block_table, bt_stride,
                 seq_lens, num_seqs, T, Hq, Hkv, D, kv_dtype};
    if (check_problem(&P) || !rows || n_rows < 0 || !out || !lse)
        return -1;
    for (int i = 0; i < n_rows; ++i) {
        int b = rows[3 * i], t = rows[3 * i + 1], h = rows[3 * i + 2];
        if (b < 0 || b >= num_seqs || t < 0 || t >= T || h < 0 || h >= Hq)
            return -1;
    }
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int i = 0; i < n_rows; ++i) {
        int b = rows[3 * i];
        failed |= attend_one(&P, b, rows[3 * i + 1], rows[3 * i + 2], 0,
                             seq_lens[b], out + (size_t)i * D, lse + i) != 0;
    }
    return failed ? -1 : 0;
}

/* Attention of one (b, t, h) restricted to the keys in [key_begin, key_end):
 * the normalised partial output and its log-sum-exp, as one split of the
 * split-KV scheme produces them.  Used to pin the log-sum-exp merge. */
int oracle_verify_attn_partial(const uint16_t *q, const void *k_pages, const void *v_pages,
                               const float *k_scale, const float *v_scale,
                               const int32_t *block_table, int bt_stride,
                               const int32_t *seq_lens, int num_seqs, int T, int Hq,
                               int Hkv, int D, int kv_dtype, int b, int t, int h,
                               int key_begin, int key_end, double *out, double *lse)
{
    problem P = {q, k_pages, v_pages, k_scale, v_scale, block_table, bt_stride,
                 seq_lens, num_seqs, T, Hq, Hkv, D, kv_dtype};
    if (check_problem(&P) || !out || !lse)
        return -1;
    if (b < 0 || b >= num_seqs || t < 0 || t >= T || h < 0 || h >= Hq)
        return -1;
    return attend_one(&P, b, t, h, key_begin, key_end, out, lse);
}
