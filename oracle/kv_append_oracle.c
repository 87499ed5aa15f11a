/*
 * CPU oracle for the KV append with quantise-on-write.  TEST INFRASTRUCTURE
 * ONLY (the tests and the benchmark's CPU-baseline leg); it shares no code,
 * header or constant with the CUDA library.
 *
 * What it computes: the verify forward stores the K and V rows of its T new
 * tokens in the paged cache before attending ("I pushed Qwen3.8-27B to 381
 * tps for a single request on a RTX 3090", "DFlash2 past 64k": int8 cache,
 * 16-token pages; "I pushed Qwen3.8-27B to 124 tps on a single request on a
 * RTX 3090", "What we had": fp8 cache).  Quantised caches keep one fp32 scale
 * per (token, kv head), the row's absmax over the largest code:
 *
 *   pos = L_b - T + t, page = block_table[b][pos / 16], slot = pos % 16
 *   x   = new row (bf16, exact in binary32)
 *   a   = max |x_d|;  s = a / qmax in binary32 (qmax 448 e4m3, 127 int8),
 *         s = 1 when a = 0
 *   y_d = x_d / s in binary32
 *   e4m3 code = round-to-nearest-even of clamp(y_d, -448, 448) (OCP e4m3:
 *               bias 7, 3 mantissa bits, subnormal step 2^-9, max 448)
 *   int8 code = clamp(round-half-even(y_d), -127, 127)
 *   int4 / int2 code = clamp(round-half-even(y_d), -qmax, qmax) with qmax 7 / 1
 *               (the int8 rule with fewer bits: the reading taken for the
 *               "KVarN 4/2-bit KV cache" bullet of the 381 tps page, which
 *               does not describe its format), packed two's complement, code
 *               d at bit (d * bits) % 8 of byte d * bits / 8
 *
 * The two divisions are binary32 on purpose: the quantised code is an integer
 * decided by a floating-point quotient, and the definition fixes that quotient
 * in single precision.  C `float` arithmetic here is IEEE binary32 with
 * round-to-nearest-even (the default mode), with no wider evaluation.
 *
 * Layouts (row-major): new rows uint16 (bf16 bits) [B, T, Hkv, D]; pages
 * [num_pages, 16, Hkv, D] of bf16 bits / e4m3 bytes / int8, or [num_pages,
 * 16, Hkv, D * bits / 8] packed bytes for int4 / int2; scales float
 * [num_pages, 16, Hkv]; block_table int32 [B, bt_stride]; seq_lens int32 [B].
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { APP_BF16 = 0, APP_E4M3 = 1, APP_INT8 = 2, APP_INT4 = 3, APP_INT2 = 4 };

static float bf16_to_float(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/* Round-to-nearest-even e4m3 code of a finite y with |y| <= 448, written from
 * the format's definition: value = (1 + m/8) 2^(E-7) for E in 1..15 (E = 15,
 * m = 7 is NaN), m/8 2^-6 for E = 0. */
uint8_t oracle_e4m3_encode(float y)
{
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    const float a = fabsf(y);
    if (a >= 448.0f)
        return sign | 0x7E;
    if (a < 0.015625f) {                  /* below 2^-6: multiples of 2^-9 */
        const float m = rintf(a * 512.0f);  /* exact scaling; m == 8 is 2^-6 = code 0x08 */
        return sign | (uint8_t)m;
    }
    int e;
    const float f = frexpf(a, &e);        /* a = f 2^e, f in [0.5, 1) */
    float m = rintf((2.0f * f - 1.0f) * 8.0f);  /* mantissa of a / 2^(e-1) in [1, 2) */
    int E = e - 1 + 7;
    if (m == 8.0f) {
        m = 0.0f;
        E += 1;
    }
    if (E > 15 || (E == 15 && m > 6.0f))
        return sign | 0x7E;
    return sign | (uint8_t)((E << 3) | (int)m);
}

int8_t oracle_int8_encode(float y)
{
    float r = rintf(y);
    if (r > 127.0f)
        r = 127.0f;
    if (r < -127.0f)
        r = -127.0f;
    return (int8_t)r;
}

/* 4-bit / 2-bit caches (the int8 rule with qmax 7 / 1): the integer code of
 * y = x / s, round-half-even, clamped to +-qmax, stored as a two's-complement
 * field at bit (d * bits) % 8 of byte d * bits / 8 of the row (the row's
 * other fields are left as they are, then overwritten in turn). */
static void append_row_packed(const uint16_t *x, int D, int bits, uint8_t *pages, float *scales, size_t row)
{
    const float qmax = (float)((1 << (bits - 1)) - 1);
    float a = 0.0f;
    for (int d = 0; d < D; ++d) {
        const float v = fabsf(bf16_to_float(x[d]));
        if (v > a)
            a = v;
    }
    const float s = a > 0.0f ? a / qmax : 1.0f;
    uint8_t *dst = pages + row * (size_t)(D * bits / 8);
    for (int d = 0; d < D; ++d) {
        float r = rintf(bf16_to_float(x[d]) / s);
        if (r > qmax)
            r = qmax;
        if (r < -qmax)
            r = -qmax;
        const int code = (int)r & ((1 << bits) - 1);
        const int bit = (d * bits) % 8;
        uint8_t *byte = dst + d * bits / 8;
        *byte = (uint8_t)((*byte & ~(((1 << bits) - 1) << bit)) | (code << bit));
    }
    scales[row] = s;
}

static void append_row(const uint16_t *x, int D, int dtype, void *pages, float *scales, size_t row)
{
    if (dtype == APP_BF16) {
        memcpy((uint16_t *)pages + row * (size_t)D, x, (size_t)D * sizeof(uint16_t));
        return;
    }
    if (dtype == APP_INT4 || dtype == APP_INT2) {
        append_row_packed(x, D, dtype == APP_INT4 ? 4 : 2, (uint8_t *)pages, scales, row);
        return;
    }
    float a = 0.0f;
    for (int d = 0; d < D; ++d) {
        const float v = fabsf(bf16_to_float(x[d]));
        if (v > a)
            a = v;
    }
    const float qmax = dtype == APP_E4M3 ? 448.0f : 127.0f;
    const float s = a > 0.0f ? a / qmax : 1.0f;
    uint8_t *dst = (uint8_t *)pages + row * (size_t)D;
    for (int d = 0; d < D; ++d) {
        float y = bf16_to_float(x[d]) / s;
        if (dtype == APP_E4M3) {
            if (y > 448.0f)
                y = 448.0f;
            if (y < -448.0f)
                y = -448.0f;
            dst[d] = oracle_e4m3_encode(y);
        } else {
            dst[d] = (uint8_t)oracle_int8_encode(y);
        }
    }
    scales[row] = s;
}

/* Returns 0, or -1 for bad arguments; rows whose position is negative or
 * whose page is outside [0, num_pages) (num_pages > 0) are skipped and
 * counted in *skipped. */
int oracle_kv_append(const uint16_t *k_new, const uint16_t *v_new, int B, int T, int Hkv, int D, int dtype,
                     void *k_pages, void *v_pages, float *k_scale, float *v_scale,
                     const int32_t *block_table, int bt_stride, const int32_t *seq_lens, int num_pages,
                     int *skipped)
{
    if (!k_new || !v_new || !k_pages || !v_pages || !block_table || !seq_lens)
        return -1;
    if (B < 1 || T < 1 || Hkv < 1 || D < 1 || bt_stride < 1 || dtype < APP_BF16 || dtype > APP_INT2)
        return -1;
    if ((dtype == APP_INT4 && D % 2) || (dtype == APP_INT2 && D % 4))
        return -1;
    if (dtype != APP_BF16 && (!k_scale || !v_scale))
        return -1;
    int n_skip = 0;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const int pos = seq_lens[b] - T + t;
            const int page = pos >= 0 ? block_table[(size_t)b * bt_stride + pos / 16] : -1;
            for (int g = 0; g < Hkv; ++g) {
                if (pos < 0 || (num_pages > 0 && (page < 0 || page >= num_pages))) {
                    n_skip += 2;
                    continue;
                }
                const size_t src = (((size_t)b * T + t) * Hkv + g) * (size_t)D;
                const size_t row = ((size_t)page * 16 + (size_t)(pos % 16)) * Hkv + g;
                append_row(k_new + src, D, dtype, k_pages, k_scale, row);
                append_row(v_new + src, D, dtype, v_pages, v_scale, row);
            }
        }
    if (skipped)
        *skipped = n_skip;
    return 0;
}
