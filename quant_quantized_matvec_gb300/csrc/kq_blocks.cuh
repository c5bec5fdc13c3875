// kq_blocks.cuh -- one super-block of one row against ntok inputs.
//
// Each function takes the block's bytes (already in registers), an accessor
// for the 256 inputs the block multiplies (x.ld(t, e) returns inputs e..e+3
// of token t, relative to the block's first input), and returns
// the block's contribution to each token's dot product.  The arithmetic is a
// fixed function of the block bytes and the inputs: every weight is first
// dequantized exactly as "Chapter 6 - The kquant family on the reference
// lane" (section 6.2) defines it -- the effective scale d*sc and min dmin*m
// are exact in f32, and fma(d*sc, code, -dmin*m) rounds once, giving the
// same f32 weight the oracle builds -- and then multiplied into one of four
// f32 accumulators chosen by the element's position within its 4-byte word.
// The four accumulators are combined as (a0 + a1) + (a2 + a3).
#pragma once

#include "kq_common.cuh"

namespace kq {

template <int NTOK>
__device__ __forceinline__ void finish(float (&acc)[NTOK][4],
                                       float (&part)[NTOK]) {
#pragma unroll
    for (int t = 0; t < NTOK; ++t)
        part[t] = (acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]);
}

// Q4_K (144 B, Figure 6.2) and Q5_K (176 B, Figure 6.4).  blk[0] holds d,
// dmin and the scale field; for Q5_K blk[1..2] hold the high-bit plane qh;
// the nibbles qs follow (8 x 16 B).  Group g (weights 64g..64g+63) reads qs
// bytes 32g..32g+31: the low nibble of byte 32g+l is weight 64g+l, the high
// nibble weight 64g+32+l.  Q5_K's fifth bit of those two weights is bit 2g,
// resp. 2g+1, of qh[l].
template <int NTOK, bool Q5, class XA>
__device__ __forceinline__ void block_q45(const uint4 (&blk)[Q5 ? 11 : 9],
                                          const XA &x, float (&part)[NTOK]) {
    constexpr int QS = Q5 ? 3 : 1;  // first uint4 of qs
    const float d = h2f(blk[0].x), dmin = h2f(blk[0].x >> 16);
    const ScaleWords sw = unpack_scale_words(blk[0].y, blk[0].z, blk[0].w);

    float acc[NTOK][4];
#pragma unroll
    for (int t = 0; t < NTOK; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t sc, m;
        scale_min(sw, 2 * g, sc, m);
        const float dl = d * u2f(sc), ml = dmin * u2f(m);
        scale_min(sw, 2 * g + 1, sc, m);
        const float dh = d * u2f(sc), mh = dmin * u2f(m);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t q = word_of(blk[QS + 2 * g + k / 4], k % 4);
            uint32_t lo = q & 0x0F0F0F0Fu;
            uint32_t hi = (q >> 4) & 0x0F0F0F0Fu;
            if (Q5) {
                const uint32_t h = word_of(blk[1 + k / 4], k % 4);
                lo |= ((h >> (2 * g)) & 0x01010101u) << 4;
                hi |= ((h >> (2 * g + 1)) & 0x01010101u) << 4;
            }
            float wl[4], wh[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wl[i] = fmaf(dl, u2f((lo >> (8 * i)) & 0xFFu), -ml);
                wh[i] = fmaf(dh, u2f((hi >> (8 * i)) & 0xFFu), -mh);
            }
#pragma unroll
            for (int t = 0; t < NTOK; ++t) {
                const float4 xl = x.ld(t, 64 * g + 4 * k);
                const float4 xh = x.ld(t, 64 * g + 32 + 4 * k);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[t][i] = fmaf(wl[i], comp(xl, i), acc[t][i]);
                    acc[t][i] = fmaf(wh[i], comp(xh, i), acc[t][i]);
                }
            }
        }
    }
    finish<NTOK>(acc, part);
}

// Q6_K (210 B, Figure 6.5), given as 52 little-endian words L[0..51] (block
// bytes 4k..4k+3) and the f16 d.  ql = L[0..31], qh = L[32..47], the sixteen
// int8 scales = L[48..51].  Half h (weights 128h..128h+127) uses ql bytes
// 64h.. and qh bytes 32h..; for l = 0..31 the weights 128h+l, +32, +64, +96
// take the low nibble of ql[64h+l], the low nibble of ql[64h+32+l], the high
// nibble of ql[64h+l], the high nibble of ql[64h+32+l], and the bit pairs
// 0-1, 2-3, 4-5, 6-7 of qh[32h+l].  Weight = d*sc[e/16]*(code-32): exact.
template <int NTOK, class XA>
__device__ __forceinline__ void block_q6(const uint32_t (&L)[52], uint32_t dbits,
                                         const XA &x, float (&part)[NTOK]) {
    const float d = h2f(dbits);
    float scl[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
        scl[j] = d * s8_to_f32(L[48 + j / 4] >> (8 * (j % 4)));

    float acc[NTOK][4];
#pragma unroll
    for (int t = 0; t < NTOK; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t qa = L[16 * h + k];      // ql[64h + 4k ..]
            const uint32_t qb = L[16 * h + 8 + k];  // ql[64h + 32 + 4k ..]
            const uint32_t qh = L[32 + 8 * h + k];  // qh[32h + 4k ..]
            uint32_t c[4];
            c[0] = (qa & 0x0F0F0F0Fu) | ((qh << 4) & 0x30303030u);
            c[1] = (qb & 0x0F0F0F0Fu) | ((qh << 2) & 0x30303030u);
            c[2] = ((qa >> 4) & 0x0F0F0F0Fu) | (qh & 0x30303030u);
            c[3] = ((qb >> 4) & 0x0F0F0F0Fu) | ((qh >> 2) & 0x30303030u);
#pragma unroll
            for (int quad = 0; quad < 4; ++quad) {
                const int e0 = 128 * h + 32 * quad + 4 * k;  // 4 weights
                const float s = scl[e0 / 16];
                float w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w[i] = s * (__int_as_float(0x4B000000u |
                                               ((c[quad] >> (8 * i)) & 0xFFu)) -
                                8388640.0f);  // code - 32, exact
#pragma unroll
                for (int t = 0; t < NTOK; ++t) {
                    const float4 xv = x.ld(t, e0);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        acc[t][i] = fmaf(w[i], comp(xv, i), acc[t][i]);
                }
            }
        }
    }
    finish<NTOK>(acc, part);
}

}  // namespace kq
