// kq_blocks.cuh -- one super-block of R rows against ntok inputs.
//
// Arithmetic ("Chapter 6 - The kquant family on the reference lane",
// section 6.2 for Q4_K, section 6.4 for Q5_K and Q6_K; "Chapter 13 - The
// QKV + gate matvec family", section 13.4.2 for the deferred-scaling form):
//
//   Q4_K / Q5_K   sum_j w_j x_j = sum_s [ (d*sc_s) * A_s - (dmin*m_s) * X_s ]
//   Q6_K          sum_j w_j x_j = sum_s (d*sc_s) * B_s
//   A_s = sum_{j in s} code_j * x_j,  B_s = sum_{j in s} (code_j - 32) * x_j,
//   X_s = sum_{j in s} x_j
//
// over the 8 sub-blocks of 32 (Q4_K, Q5_K) or 16 sub-blocks of 16 (Q6_K).
// The inputs come as the fixed-point records of kq_xrec.cuh (x_j = X_j * u
// per group of 32, X_j split into three bytes), so A_s and B_s are
//   u * ((S2 * 256 + S1) * 256 + S0),  S_l = sum_{j in s} code_j * b_l(X_j)
// with S_l exact integer byte dot products (dp4a, four codes a step).  Codes
// stay packed four to a word as they sit in the block, masked (and, for
// Q5_K and Q6_K, merged with their high bits) in place:
//   Q4_K  low nibbles as codes; high nibbles left at bits 4..7 (16 * code),
//         the factor 1/16 taken into d of the odd sub-blocks
//   Q5_K  low codes in bits 0..4; high codes in bits 3..7 (8 * code), 1/8
//         taken into d of the odd sub-blocks
//   Q6_K  codes in bits 0..5; the offset -32 enters through the records'
//         starting values -32 * sum b_l, so the limb sums stay exact
// d*sc and dmin*m are exact in f32; each sub-block adds one rounded term
// (d*sc_s * u) * A_s to the row's f32 sum, in sub-block order, and the
// Q4_K / Q5_K min term sum_s (dmin*m_s) * X_s is subtracted last.
//
// Each row's sequence of operations is fixed by the format and ntok alone
// (R only interleaves independent rows), so a block's contribution is the
// same function of its bytes and its inputs in every kernel.
#pragma once

#include "kq_common.cuh"
#include "kq_xrec.cuh"

namespace kq {

// ------------------------------------------------------------ primitives
// c + the sum of the four byte products a_i * b_i: a unsigned; b unsigned
// (uu) or signed (us).
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// (a & m) | b in one three-input logic instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t b) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(b));
    return d;
}
// (a & m) | (b & ~m) in one three-input logic instruction.
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
    return d;
}
// A 32-bit constant in a register the compiler cannot fold into an
// instruction (keeps each mask step a single logic instruction).
__device__ __forceinline__ uint32_t reg_u32(uint32_t c) {
    uint32_t v;
    asm("mov.b32 %0, %1;" : "=r"(v) : "r"(c));
    return v;
}
// Three exact limb sums -> (S2 * 256 + S1) * 256 + S0 in f32: one rounding
// in each conversion and one in the fma.  |S2 * 256 + S1| < 2^31 for every
// format (at most 32 codes below 256 against bytes below 256).
__device__ __forceinline__ float limbs_f32(int s0, int s1, int s2) {
    return fmaf(__int2float_rn(s2 * 256 + s1), 256.0f, __int2float_rn(s0));
}

// ------------------------------------------------------------ records
// Accessor of the input records (kq_xrec.cuh) of one super-block column:
// p = its record for token 0, tstride = bytes between tokens.  GLOBAL
// selects read-only global loads, else plain (shared-memory) loads.
template <bool GLOBAL>
struct Rec {
    const uint8_t *p;
    int tstride;
    template <class T>
    __device__ __forceinline__ T ld(int off) const {
        const T *q = reinterpret_cast<const T *>(p + off);
        if (GLOBAL) return __ldg(q);
        return *q;
    }
    // plane l (0..2), inputs e..e+15 (e a multiple of 16)
    __device__ __forceinline__ uint4 plane(int t, int l, int e) const {
        return ld<uint4>(t * tstride + 256 * l + e);
    }
    __device__ __forceinline__ float u1(int t, int g) const {
        return ld<float>(t * tstride + kRecU + 4 * g);
    }
    __device__ __forceinline__ float2 u2(int t, int g2) const {  // groups 2*g2, 2*g2+1
        return ld<float2>(t * tstride + kRecU + 8 * g2);
    }
    __device__ __forceinline__ void sums8(int t, float (&o)[8]) const {
        const float4 a = ld<float4>(t * tstride + kRecSums);
        const float4 b = ld<float4>(t * tstride + kRecSums + 16);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
    __device__ __forceinline__ int4 start6(int t, int s) const {  // Q6_K sub-block s
        return ld<int4>(t * tstride + kRecSums + 16 * s);
    }
};

// ------------------------------------------------------------ scales
// Byte k (a value below 256) of w as the float 2^23 + value.
__device__ __forceinline__ float magic_byte(uint32_t w, int k, uint32_t m23) {
    return __uint_as_float(__byte_perm(w, m23, 0x7650 | k));
}

// Header of a Q4_K / Q5_K block (d, dmin, the 12-byte scale field), decoded
// where it is used.  d*sc and dmin*m are exact: with F = 2^23 + v (v below
// 64), fma(d, F, -d * 2^23) = d * v, which has at most 17 significant bits.
// dh = d * 2^-k is the d of the odd sub-blocks, whose codes sit k bits up.
struct Q45Head {
    ScaleWords sw;
    float d, nd, dh, ndh, dmin, ndm;  // nd = -d * 2^23 and so on
    Q45Head() = default;
    __device__ __forceinline__ Q45Head(const uint4 &h, float hscale) {
        d = h2f(h.x);
        dmin = h2f(h.x >> 16);
        dh = d * hscale;
        nd = -d * 8388608.0f;
        ndh = -dh * 8388608.0f;
        ndm = -dmin * 8388608.0f;
        sw = unpack_scale_words(h.y, h.z, h.w);
    }
    // (d*sc_{2g}, dh*sc_{2g+1}); g may be a runtime value
    __device__ __forceinline__ float2 scale_pair(int g, uint32_t m23) const {
        const uint32_t w = g < 2 ? sw.sc_lo : sw.sc_hi;
        const uint32_t k = 2u * (uint32_t)(g & 1);
        const float f0 = __uint_as_float(__byte_perm(w, m23, 0x7650u | k));
        const float f1 = __uint_as_float(__byte_perm(w, m23, 0x7650u | (k + 1u)));
        return __ffma2_rn(make_float2(d, dh), make_float2(f0, f1), make_float2(nd, ndh));
    }
    // (dmin*m_k, dmin*m_{k+4}) for k = 0..3
    __device__ __forceinline__ float2 min_pair(int k, uint32_t m23) const {
        return __ffma2_rn(make_float2(dmin, dmin),
                          make_float2(magic_byte(sw.m_lo, k, m23), magic_byte(sw.m_hi, k, m23)),
                          make_float2(ndm, ndm));
    }
};

// Min term sum_s (dmin*m_s) * X_s in sub-block order.
template <class XR>
__device__ __forceinline__ float q45_min_term(const Q45Head &hd, const XR &xr, int t,
                                              uint32_t m23) {
    float dm[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 p = hd.min_pair(k, m23);
        dm[k] = p.x;
        dm[k + 4] = p.y;
    }
    float xs[8];
    xr.sums8(t, xs);
    float mt = 0.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s) mt = fmaf(dm[s], xs[s], mt);
    return mt;
}

// ------------------------------------------------------------ byte sources
// B.v4(i): the i-th 16-byte chunk of a Q4_K / Q5_K block (16-byte aligned).
struct BlockShared {
    const uint4 *p;
    __device__ __forceinline__ uint4 v4(int i) const { return p[i]; }
};
struct BlockGlobal {
    const uint4 *p;
    __device__ __forceinline__ uint4 v4(int i) const { return __ldg(p + i); }
};

// Q6_K blocks are 2-byte aligned.  W.words4(j, o) gives block words
// j..j+3 (bytes 4j..4j+15), W.dbits() the f16 d at bytes 208..209.
// SHIFTED: the block starts 2 bytes past a 4-byte boundary and a = its
// start - 2; else a = its start, 4-byte aligned.  No byte outside the
// block is read.
template <bool SHIFTED, bool GLOBAL>
struct Q6Words {
    const uint8_t *a;
    __device__ __forceinline__ uint32_t w(int i) const {
        const uint32_t *q = reinterpret_cast<const uint32_t *>(a + 4 * i);
        if (GLOBAL) return __ldg(q);
        return *q;
    }
    __device__ __forceinline__ void words4(int j, uint32_t (&o)[4]) const {
        if (SHIFTED) {
            uint32_t r[5];
#pragma unroll
            for (int i = 0; i < 5; ++i) r[i] = w(j + i);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(r[i], r[i + 1], 16);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = w(j + i);
        }
    }
    __device__ __forceinline__ uint32_t dbits() const {
        if (SHIFTED) return w(52) >> 16;
        const unsigned short *q = reinterpret_cast<const unsigned short *>(a + 208);
        if (GLOBAL) return __ldg(q);
        return *q;
    }
};

// ------------------------------------------------------------ Q4_K / Q5_K
// Q4_K: chunk 0 header, chunks 1..8 qs (group g: chunks 1 + 2g, 2 + 2g).
// Q5_K: chunk 0 header, chunks 1..2 qh, chunks 3..10 qs.
// Group g = weights 64g..64g+63: byte 32g + l of qs holds weight 64g + l
// (low nibble, sub-block 2g) and 64g + 32 + l (high nibble, 2g + 1); for
// Q5_K bit 2g of qh[l] is the fifth bit of weight 64g + l and bit 2g + 1
// that of weight 64g + 32 + l.  R rows share the block column's inputs.
template <int NTOK, bool Q5, int R, class BS, class XR>
__device__ __forceinline__ void block_q45(const BS (&B)[R], const XR &xr,
                                          float (&part)[R][NTOK]) {
    const uint32_t m23 = reg_u32(0x4B000000u);
    const uint32_t nib = reg_u32(0x0F0F0F0Fu);
    const uint32_t hmask = reg_u32(Q5 ? 0x78787878u : 0xF0F0F0F0u);
    Q45Head hd[R];
    uint32_t qh[R][8];
    float acc[R][NTOK];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        hd[r] = Q45Head(B[r].v4(0), Q5 ? 0.125f : 0.0625f);
        if (Q5) {
            const uint4 a = B[r].v4(1), b = B[r].v4(2);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qh[r][k] = word_of(a, k);
                qh[r][4 + k] = word_of(b, k);
            }
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t) acc[r][t] = 0.0f;
    }
    constexpr int QS = Q5 ? 3 : 1;
    // one token: the four groups fully unrolled, for independent work to
    // interleave (measured 3% faster); more tokens keep the loop, whose
    // unrolled form spills
#pragma unroll(NTOK == 1 ? 4 : 1)
    for (int g = 0; g < 4; ++g) {
        uint32_t lo[R][8], hi[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint4 a = B[r].v4(QS + 2 * g), b = B[r].v4(QS + 2 * g + 1);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t w = word_of(k < 4 ? a : b, k & 3);
                if (Q5) {
                    const uint32_t hs = qh[r][k] >> (2 * g);
                    lo[r][k] = and_or(w, nib, (hs & 0x01010101u) << 4);
                    hi[r][k] = and_or(w >> 1, hmask, (hs & 0x02020202u) << 6);
                } else {
                    lo[r][k] = w & nib;
                    hi[r][k] = w & hmask;
                }
            }
        }
        float2 ds[R];
#pragma unroll
        for (int r = 0; r < R; ++r) ds[r] = hd[r].scale_pair(g, m23);
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
            int sl[R][3], sh[R][3];
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int l = 0; l < 3; ++l) sl[r][l] = sh[r][l] = 0;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                uint4 xl[3], xh[3];
#pragma unroll
                for (int l = 0; l < 3; ++l) {
                    xl[l] = xr.plane(t, l, 64 * g + 16 * m);
                    xh[l] = xr.plane(t, l, 64 * g + 32 + 16 * m);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t cl = lo[r][4 * m + k], ch = hi[r][4 * m + k];
                        sl[r][0] = dp4a_uu(cl, word_of(xl[0], k), sl[r][0]);
                        sl[r][1] = dp4a_uu(cl, word_of(xl[1], k), sl[r][1]);
                        sl[r][2] = dp4a_us(cl, word_of(xl[2], k), sl[r][2]);
                        sh[r][0] = dp4a_uu(ch, word_of(xh[0], k), sh[r][0]);
                        sh[r][1] = dp4a_uu(ch, word_of(xh[1], k), sh[r][1]);
                        sh[r][2] = dp4a_us(ch, word_of(xh[2], k), sh[r][2]);
                    }
            }
            const float2 u = xr.u2(t, g);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float2 c = __fmul2_rn(ds[r], u);
                acc[r][t] = fmaf(c.x, limbs_f32(sl[r][0], sl[r][1], sl[r][2]), acc[r][t]);
                acc[r][t] = fmaf(c.y, limbs_f32(sh[r][0], sh[r][1], sh[r][2]), acc[r][t]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NTOK; ++t) part[r][t] = acc[r][t] - q45_min_term(hd[r], xr, t, m23);
}

// ------------------------------------------------------------------ Q6_K
// ql = words 0..31, qh = words 32..47, int8 scales = words 48..51, f16 d at
// bytes 208..209.  Half h (weights 128h..128h+127) reads ql bytes 64h.. and
// qh bytes 32h..; for l = 0..31 the weights 128h+l, +32, +64, +96
// (quadrants 0..3) take the low nibble of ql[64h+l], the low nibble of
// ql[64h+32+l], the high nibble of ql[64h+l], the high nibble of
// ql[64h+32+l], and bit pairs 0-1, 2-3, 4-5, 6-7 of qh[32h+l] as bits 4-5.
// Step `it` = 2h + kh takes words k = 4kh..4kh+3 of the half: sub-block
// 8h + 2q + kh of each quadrant q.  All R rows' blocks share one alignment.
template <int NTOK, int R, class WS, class XR>
__device__ __forceinline__ void block_q6k(const WS (&W)[R], const XR &xr, float (&part)[R][NTOK]) {
    const uint32_t m23 = reg_u32(0x4B000000u);
    const uint32_t nib = reg_u32(0x0F0F0F0Fu);
    float d[R];
    uint32_t scw[R][4];
    float acc[R][NTOK];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        d[r] = h2f(W[r].dbits());
        W[r].words4(48, scw[r]);
        // signed scale bytes biased to 0..255 for the magic-float decode
#pragma unroll
        for (int i = 0; i < 4; ++i) scw[r][i] ^= 0x80808080u;
#pragma unroll
        for (int t = 0; t < NTOK; ++t) acc[r][t] = 0.0f;
    }
#pragma unroll 1
    for (int it = 0; it < 4; ++it) {
        const int h = it >> 1, kh = it & 1;
        uint32_t c[R][4][4];  // [row][quadrant][word]
        float dsc[R][4];      // d * sc of sub-block 8h + 2q + kh
#pragma unroll
        for (int r = 0; r < R; ++r) {
            uint32_t qa[4], qb[4], qq[4];
            W[r].words4(16 * h + 4 * kh, qa);
            W[r].words4(16 * h + 8 + 4 * kh, qb);
            W[r].words4(32 + 8 * h + 4 * kh, qq);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t qm = qq[k] & 0x33333333u, qn = qq[k] & 0xCCCCCCCCu;
                c[r][0][k] = bitsel(qa[k], qm << 4, nib);
                c[r][1][k] = bitsel(qb[k], qn << 2, nib);
                c[r][2][k] = bitsel(qa[k] >> 4, qm, nib);
                c[r][3][k] = bitsel(qb[k] >> 4, qn >> 2, nib);
            }
            // sub-block 8h + 2q + kh: scale byte (2q + kh) & 3 of word 2h + q / 2,
            // d * (F - (2^23 + 128)) with F = 2^23 + (sc + 128)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t wsc = h ? scw[r][2 + (q >> 1)] : scw[r][q >> 1];
                const float f = __uint_as_float(
                    __byte_perm(wsc, m23, 0x7650u | (uint32_t)(2 * (q & 1) + kh)));
                dsc[r][q] = d[r] * (f - 8388736.0f);
            }
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int4 st = xr.start6(t, 8 * h + 2 * q + kh);
                int s[R][3];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    s[r][0] = st.x;
                    s[r][1] = st.y;
                    s[r][2] = st.z;
                }
                const int e = 128 * h + 32 * q + 16 * kh;
                const uint4 x0 = xr.plane(t, 0, e), x1 = xr.plane(t, 1, e), x2 = xr.plane(t, 2, e);
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        s[r][0] = dp4a_uu(c[r][q][k], word_of(x0, k), s[r][0]);
                        s[r][1] = dp4a_uu(c[r][q][k], word_of(x1, k), s[r][1]);
                        s[r][2] = dp4a_us(c[r][q][k], word_of(x2, k), s[r][2]);
                    }
                const float u = xr.u1(t, 4 * h + q);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    acc[r][t] = fmaf(dsc[r][q] * u, limbs_f32(s[r][0], s[r][1], s[r][2]), acc[r][t]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NTOK; ++t) part[r][t] = acc[r][t];
}

}  // namespace kq
