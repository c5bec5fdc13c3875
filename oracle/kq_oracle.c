/*
 * kq_oracle.c -- plain CPU reference for the K-quant matvec.
 *
 * TEST INFRASTRUCTURE ONLY (see kq_oracle.h).  Compiled with gcc
 * -O2 -ffp-contract=off so that every f32 operation written below rounds
 * exactly where it is written, on x86-64 and on aarch64 alike.
 *
 * No blocking, fusion or reordering: a row is dequantized block by block,
 * then each token's dot product is summed in f64 in element order.
 */
#include "kq_oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>

/* Figure 6.1 of "Chapter 6 - The kquant family": bytes per 256 elements. */
int kqo_block_bytes(int fmt)
{
    switch (fmt) {
    case KQO_Q4_K: return 144;  /* 2 + 2 + 12 + 128           (Figure 6.2) */
    case KQO_Q5_K: return 176;  /* 2 + 2 + 12 + 32 + 128      (Figure 6.4) */
    case KQO_Q6_K: return 210;  /* 128 + 64 + 16 + 2          (Figure 6.5) */
    default: return -1;
    }
}

/*
 * Reading R3: the f16 header fields are IEEE 754 binary16 -- 1 sign bit,
 * 5 exponent bits with bias 15, 10 fraction bits; exponent 0 is the
 * subnormal range fraction * 2^-24, exponent 31 is inf / NaN.  Written from
 * that definition; every binary16 value is exact in f32, so the double
 * computed here converts to float without rounding.
 */
float kqo_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = (f == 0) ? INFINITY : NAN;
    else
        v = ldexp(1024.0 + (double)f, e - 25);  /* (1 + f/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/*
 * Section 6.2 / Figure 6.3: twelve bytes hold eight 6-bit scales and eight
 * 6-bit mins.  Sub-blocks 0..3 keep both in the low six bits of bytes j and
 * j+4.  Sub-blocks 4..7 take their low four bits from byte j+4 (scale: low
 * nibble, min: high nibble) and their top two bits from the spare top bits
 * of bytes j-4 (scale) and j (min).
 */
void kqo_scale_min_k4(const uint8_t scales[12], int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

static uint16_t le16(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

/*
 * Q4_K (section 6.2, Figure 6.2): d at byte 0, dmin at byte 2, the scale
 * field at 4..15, 128 bytes of nibbles at 16..143.  The 256 weights form
 * four groups of 64; group g reads qs bytes 32g..32g+31.  The low nibble of
 * byte 32g+l is weight 64g+l (sub-block 2g), the high nibble is weight
 * 64g+32+l (sub-block 2g+1).  Weight = (d*sc) * nibble - (dmin*m), in f32.
 *
 * Q5_K (section 6.4, Figure 6.4) is the same with a fifth bit per weight
 * from the 32-byte plane qh at 16..47; the nibbles move to 48..175.
 * Reading R1 (the pages print the formula w = d*sc*(nibble | qh_bit<<4) -
 * dmin*m but not which bit): bit 2g of qh[l] belongs to weight 64g+l and
 * bit 2g+1 to weight 64g+32+l -- the same low/high pairing as the nibbles.
 */
static void dequant_q45(const uint8_t *b, int has_qh, float *out)
{
    const float d = kqo_f16_to_f32(le16(b + 0));
    const float dmin = kqo_f16_to_f32(le16(b + 2));
    const uint8_t *scales = b + 4;
    const uint8_t *qh = b + 16;
    const uint8_t *qs = b + (has_qh ? 48 : 16);

    for (int g = 0; g < 4; ++g) {
        int sc_lo, m_lo, sc_hi, m_hi;
        kqo_scale_min_k4(scales, 2 * g, &sc_lo, &m_lo);
        kqo_scale_min_k4(scales, 2 * g + 1, &sc_hi, &m_hi);
        const float d_lo = d * (float)sc_lo, min_lo = dmin * (float)m_lo;
        const float d_hi = d * (float)sc_hi, min_hi = dmin * (float)m_hi;
        for (int l = 0; l < 32; ++l) {
            const uint8_t q = qs[32 * g + l];
            int code_lo = q & 15;
            int code_hi = q >> 4;
            if (has_qh) {
                code_lo |= ((qh[l] >> (2 * g)) & 1) << 4;
                code_hi |= ((qh[l] >> (2 * g + 1)) & 1) << 4;
            }
            out[64 * g + l] = d_lo * (float)code_lo - min_lo;
            out[64 * g + 32 + l] = d_hi * (float)code_hi - min_hi;
        }
    }
}

/*
 * Q6_K (section 6.4, Figure 6.5): ql (low four bits of every code, two per
 * byte) at 0..127, qh (two high bits of four codes per byte) at 128..191,
 * sixteen int8 sub-block scales at 192..207 (one per 16 weights), f16 d at
 * 208..209.  Code = (low nibble | two high bits << 4), 0..63; weight =
 * d * sc[e/16] * (code - 32).
 *
 * Reading R2 (the pages name the four-way pairing but not its order): the
 * block is two halves of 128 weights, half h using ql[64h..64h+63] and
 * qh[32h..32h+31].  For l = 0..31 the byte qh[32h+l] carries, from its low
 * bits up, the high bits of weights 128h+l, +32, +64, +96; those weights
 * take their low bits from the low nibble of ql[64h+l], the low nibble of
 * ql[64h+32+l], the high nibble of ql[64h+l] and the high nibble of
 * ql[64h+32+l], in that order.
 */
static void dequant_q6(const uint8_t *b, float *out)
{
    const uint8_t *ql = b;
    const uint8_t *qh = b + 128;
    const int8_t *sc = (const int8_t *)(b + 192);
    const float d = kqo_f16_to_f32(le16(b + 208));

    for (int h = 0; h < 2; ++h) {
        const uint8_t *L = ql + 64 * h;
        const uint8_t *H = qh + 32 * h;
        for (int l = 0; l < 32; ++l) {
            const int e = 128 * h + l;
            int code[4];
            code[0] = (L[l] & 15) | (((H[l] >> 0) & 3) << 4);
            code[1] = (L[l + 32] & 15) | (((H[l] >> 2) & 3) << 4);
            code[2] = (L[l] >> 4) | (((H[l] >> 4) & 3) << 4);
            code[3] = (L[l + 32] >> 4) | (((H[l] >> 6) & 3) << 4);
            for (int k = 0; k < 4; ++k) {
                const int idx = e + 32 * k;
                const float scale = d * (float)sc[idx / 16];
                out[idx] = scale * (float)(code[k] - 32);
            }
        }
    }
}

int kqo_dequant_block(int fmt, const uint8_t *block, float out[256])
{
    switch (fmt) {
    case KQO_Q4_K: dequant_q45(block, 0, out); return 0;
    case KQO_Q5_K: dequant_q45(block, 1, out); return 0;
    case KQO_Q6_K: dequant_q6(block, out); return 0;
    default: return -1;
    }
}

/* Rows are contiguous runs of super-blocks (section 13.3; section 6.6). */
int kqo_dequant_row(int fmt, const uint8_t *W, int64_t cols, int64_t row,
                    float *out)
{
    const int bb = kqo_block_bytes(fmt);
    if (bb < 0 || cols <= 0 || cols % 256 != 0 || row < 0)
        return -1;
    const int64_t nb = cols / 256;
    const uint8_t *r = W + row * nb * bb;
    for (int64_t b = 0; b < nb; ++b)
        kqo_dequant_block(fmt, r + b * bb, out + b * 256);
    return 0;
}

/* One dot product in f64, in element order; S is the sum of |products|. */
static void dot_f64(const float *w, const float *x, int64_t n, double *y,
                    double *S)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double p = (double)w[j] * (double)x[j];
        acc += p;
        mag += fabs(p);
    }
    *y = acc;
    *S = mag;
}

void kqo_matvec_f32(const float *W, int64_t rows, int64_t cols,
                    const float *x, int ntok, double *y, double *S)
{
    for (int t = 0; t < ntok; ++t)
        for (int64_t i = 0; i < rows; ++i)
            dot_f64(W + i * cols, x + t * cols, cols, &y[t * rows + i],
                    &S[t * rows + i]);
}

int kqo_matvec_rows(int fmt, const uint8_t *W, int64_t rows, int64_t cols,
                    const float *x, int ntok, const int64_t *row_idx,
                    int64_t n, double *y, double *S)
{
    if (kqo_block_bytes(fmt) < 0 || cols <= 0 || cols % 256 != 0 ||
        rows <= 0 || ntok < 1 || n < 0)
        return -1;
    /* A row of cols f32 weights, dequantized once and used for every token. */
    float *wrow = (float *)malloc((size_t)cols * sizeof(float));
    if (!wrow)
        return -1;
    for (int64_t k = 0; k < n; ++k) {
        const int64_t i = row_idx ? row_idx[k] : k;
        if (i < 0 || i >= rows) {
            free(wrow);
            return -1;
        }
        kqo_dequant_row(fmt, W, cols, i, wrow);
        for (int t = 0; t < ntok; ++t)
            dot_f64(wrow, x + (int64_t)t * cols, cols, &y[t * n + k],
                    &S[t * n + k]);
    }
    free(wrow);
    return 0;
}
