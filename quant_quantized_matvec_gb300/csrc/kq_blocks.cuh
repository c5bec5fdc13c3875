// kq_blocks.cuh -- one super-block of one row against ntok inputs.
//
// Arithmetic ("Chapter 6 - The kquant family on the reference lane",
// section 6.2 for Q4_K, section 6.4 for Q5_K and Q6_K; "Chapter 13 - The
// QKV + gate matvec family", section 13.4.2 for the deferred-scaling form):
//
//   Q4_K / Q5_K   sum_j w_j x_j = sum_s [ (d*sc_s) * A_s - (dmin*m_s) * X_s ]
//                 A_s = sum_{j in s} code_j * x_j,  X_s = sum_{j in s} x_j
//   Q6_K          sum_j w_j x_j = sum_s (d*sc_s) * B_s
//                 B_s = sum_{j in s} (code_j - 32) * x_j
//
// over the 8 sub-blocks of 32 (Q4_K, Q5_K) or 16 sub-blocks of 16 (Q6_K).
// d*sc and dmin*m are exact in f32.  X_s is the sum of the sub-block's 32
// inputs in element order, computed once per input vector.
//
// Each product code_j * x_j is formed without an integer-to-float
// conversion.  A code sitting at bit position o of a 32-bit word is OR-ed,
// unshifted, into the mantissa of 1.0f: F = 1 + code * 2^(o-23).  F - 1 (or
// F - (1 + 32 * 2^(o-23)) for Q6_K's offset codes) is exact -- both operands
// lie in [1, 2) -- and equals code * 2^(o-23).  The inputs are stored
// pre-multiplied by 2^(23-o) for the position their code occupies (an exact
// power-of-two scaling), so the f32 product of the two is exactly the f32
// product code * x rounded once.  Pairs of weights go through the packed
// f32x2 add and fma of sm_100+ (__fadd2_rn, __ffma2_rn).
//
// The order of every operation is fixed by the format alone, so a block's
// contribution is a fixed function of its bytes and its inputs.
#pragma once

#include "kq_common.cuh"

namespace kq {

constexpr uint32_t kOne = 0x3F800000u;  // 1.0f

// Exponent k = 23 - o of the input scaling 2^k applied to element e
// (0..255) of a block, o being the bit position its code occupies in the
// word the float is built from (always inside the 23 mantissa bits):
//   Q4_K:        low nibbles {0, 8, 16, 12}[e & 3], high nibbles
//                {4, 12, 8, 16}[e & 3] (high half of a 64-weight group)
//   Q5_K, Q6_K:  {0, 8, 16, ((e >> 5) & 1) ? 16 : 0}[e & 3]
__host__ __device__ constexpr int xscale_pos(bool q4, int e) {
    return q4 ? (((e >> 5) & 1) ? ((e & 3) == 0 ? 4 : (e & 3) == 1 ? 12 : (e & 3) == 2 ? 8 : 16)
                                : ((e & 3) == 0 ? 0 : (e & 3) == 1 ? 8 : (e & 3) == 2 ? 16 : 12))
              : ((e & 3) == 0 ? 0 : (e & 3) == 1 ? 8 : (e & 3) == 2 ? 16 : (((e >> 5) & 1) ? 16 : 0));
}
__host__ __device__ constexpr int xscale_exp(bool q4, int e) { return 23 - xscale_pos(q4, e); }
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }

__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b) {
    return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// (a & m) | c in one three-input logic instruction.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
    return d;
}
// 1.0f in a register the compiler cannot fold: keeps each code-to-float
// step a single logic instruction with the mask as its only immediate.
__device__ __forceinline__ uint32_t reg_one() {
    uint32_t v;
    asm("mov.b32 %0, 0x3F800000;" : "=r"(v));
    return v;
}
__device__ __forceinline__ float reg_f32(float c) {
    float v;
    asm("mov.b32 %0, %1;" : "=f"(v) : "f"(c));
    return v;
}
// The float 1 + code * 2^(o-23) for the code under mask m (bits o..).
__device__ __forceinline__ uint32_t fone(uint32_t a, uint32_t m, uint32_t one) {
    return and_or(a, m, one);
}

// Input accessors.  xs4(t, e): the scaled inputs e..e+3 of token t (e a
// multiple of 4, relative to the block); xsum(t, s): X_s of sub-block s.
struct XSharedS {
    const float *x;  // scaled inputs of this block, token 0 (shared memory)
    int xplane;      // floats between token planes
    const float *s;  // sub-block sums of this block, token 0 (shared memory)
    int splane;
    __device__ __forceinline__ float4 xs4(int t, int e) const {
        return *reinterpret_cast<const float4 *>(x + t * xplane + e);
    }
    __device__ __forceinline__ void xsum8(int t, float (&o)[8]) const {
        const float4 a = *reinterpret_cast<const float4 *>(s + t * splane);
        const float4 b = *reinterpret_cast<const float4 *>(s + t * splane + 4);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    }
};

// Sum of 32 consecutive inputs in element order (the definition of X_s).
__device__ __forceinline__ float sum32(const float *p) {
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        const float4 v = ldg_f4(p + j);
        acc += v.x;
        acc += v.y;
        acc += v.z;
        acc += v.w;
    }
    return acc;
}

template <bool Q4>
struct XGlobalS {  // unscaled inputs in global memory, scaled on the fly
    const float *p;
    int64_t plane;
    __device__ __forceinline__ float4 xs4(int t, int e) const {
        float4 v = ldg_f4(p + t * plane + e);
        v.x *= pow2f(xscale_exp(Q4, e));
        v.y *= pow2f(xscale_exp(Q4, e + 1));
        v.z *= pow2f(xscale_exp(Q4, e + 2));
        v.w *= pow2f(xscale_exp(Q4, e + 3));
        return v;
    }
    __device__ __forceinline__ void xsum8(int t, float (&o)[8]) const {
#pragma unroll
        for (int s = 0; s < 8; ++s) o[s] = sum32(p + t * plane + 32 * s);
    }
};

// ------------------------------------------------------------------ scales
// Byte k (a value below 256) of w as the float 2^23 + value.
__device__ __forceinline__ float magic_byte(uint32_t w, int k, uint32_t m23) {
    return __uint_as_float(__byte_perm(w, m23, 0x7650 | k));
}

// Scales and mins of a Q4_K / Q5_K block, decoded where they are used.
// d*sc and dmin*m are exact: with F = 2^23 + v (v below 64),
// fma(d, F, -d * 2^23) = d * v, which has at most 17 significant bits.
struct Q45Head {
    ScaleWords sw;
    float d, nd, dmin, ndm;  // nd = -d * 2^23, ndm = -dmin * 2^23
    Q45Head() = default;
    __device__ __forceinline__ explicit Q45Head(const uint4 &h) {
        d = h2f(h.x);
        dmin = h2f(h.x >> 16);
        nd = -d * 8388608.0f;
        ndm = -dmin * 8388608.0f;
        sw = unpack_scale_words(h.y, h.z, h.w);
    }
    // (d*sc_{2g}, d*sc_{2g+1}); g may be a runtime value
    __device__ __forceinline__ float2 scale_pair(int g, uint32_t m23) const {
        const uint32_t w = g < 2 ? sw.sc_lo : sw.sc_hi;
        const uint32_t k = 2u * (uint32_t)(g & 1);
        const float f0 = __uint_as_float(__byte_perm(w, m23, 0x7650u | k));
        const float f1 = __uint_as_float(__byte_perm(w, m23, 0x7650u | (k + 1u)));
        return __ffma2_rn(make_float2(d, d), make_float2(f0, f1), make_float2(nd, nd));
    }
    // (dmin*m_k, dmin*m_{k+4}) for k = 0..3
    __device__ __forceinline__ float2 min_pair(int k, uint32_t m23) const {
        return __ffma2_rn(make_float2(dmin, dmin),
                          make_float2(magic_byte(sw.m_lo, k, m23), magic_byte(sw.m_hi, k, m23)),
                          make_float2(ndm, ndm));
    }
};

// Min term sum_s (dmin*m_s) * X_s in sub-block order.
template <class XA>
__device__ __forceinline__ float q45_min_term(const Q45Head &hd, const XA &x, int t,
                                              uint32_t m23) {
    float dm[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 p = hd.min_pair(k, m23);
        dm[k] = p.x;
        dm[k + 4] = p.y;
    }
    float xsb[8];
    x.xsum8(t, xsb);
    float mt = 0.0f;
#pragma unroll
    for (int sb = 0; sb < 8; ++sb) mt = fmaf(dm[sb], xsb[sb], mt);
    return mt;
}

// Sum of a sub-block's two accumulator pairs: (a0.x + a1.x) + (a0.y + a1.y).
__device__ __forceinline__ float pair_sum(float2 a0, float2 a1) {
    const float2 s = __fadd2_rn(a0, a1);
    return s.x + s.y;
}

// (a & m) | (b & ~m) in one three-input logic instruction.
__device__ __forceinline__ uint32_t bitsel(uint32_t a, uint32_t b, uint32_t m) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(d) : "r"(a), "r"(b), "r"(m));
    return d;
}

// Block byte sources for kq_blocks: B.v4(i) is the i-th 16-byte chunk of a
// Q4_K / Q5_K block (16-byte aligned in shared or global memory).
struct BlockShared {
    const uint4 *p;
    __device__ __forceinline__ uint4 v4(int i) const { return p[i]; }
};
struct BlockGlobal {
    const uint4 *p;
    __device__ __forceinline__ uint4 v4(int i) const { return __ldg(p + i); }
};

// One 32-byte qs run (eight words, 64 weights of group g) of a Q4_K block,
// for R rows that share the same inputs: the low nibble of byte 32g+l is
// weight 64g+l (sub-block 2g), the high nibble weight 64g+32+l (2g+1).
// al / ah accumulate code * x of the two sub-blocks, per row and token, as
// two f32x2 chains each.
template <int NTOK, int R, class XA>
__device__ __forceinline__ void q4_group(const uint4 (&w0)[R], const uint4 (&w1)[R], const XA &x,
                                         int e0, uint32_t one, float2 m1,
                                         float2 (&al)[R][NTOK][2], float2 (&ah)[R][NTOK][2]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float2 l01[R], l23[R], h01[R], h23[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t q = word_of(k < 4 ? w0[r] : w1[r], k % 4);
            // q >> 12 brings the high nibble of byte 2 to bits 8..11 and byte
            // 3's nibbles to bits 12..19 (bit 23 is the exponent's)
            const uint32_t q3 = q >> 12;
            l01[r] = __fadd2_rn(f2(fone(q, 0xFu, one), fone(q, 0xF00u, one)), m1);
            l23[r] = __fadd2_rn(f2(fone(q, 0xF0000u, one), fone(q3, 0xF000u, one)), m1);
            h01[r] = __fadd2_rn(f2(fone(q, 0xF0u, one), fone(q, 0xF000u, one)), m1);
            h23[r] = __fadd2_rn(f2(fone(q3, 0xF00u, one), fone(q3, 0xF0000u, one)), m1);
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
            const float4 xl = x.xs4(t, e0 + 4 * k);
            const float4 xh = x.xs4(t, e0 + 32 + 4 * k);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                al[r][t][0] = __ffma2_rn(l01[r], make_float2(xl.x, xl.y), al[r][t][0]);
                al[r][t][1] = __ffma2_rn(l23[r], make_float2(xl.z, xl.w), al[r][t][1]);
                ah[r][t][0] = __ffma2_rn(h01[r], make_float2(xh.x, xh.y), ah[r][t][0]);
                ah[r][t][1] = __ffma2_rn(h23[r], make_float2(xh.z, xh.w), ah[r][t][1]);
            }
        }
    }
}

// Q5_K: the same with the fifth bit of weight 64g+l (bit 2g of qh[l]) and of
// weight 64g+32+l (bit 2g+1).  Codes are assembled four at a time with one
// bit-select: nibble in bits 0..3 of each byte, the high bit shifted into
// bit 4 (bits 5..7 of a byte hold other qh bits and are masked off when the
// float is built).  qh words are shifted right by 2g first so that every
// group uses the shifts of group 0.
template <int NTOK, int R, class XA>
__device__ __forceinline__ void q5_group(const uint4 (&w0)[R], const uint4 (&w1)[R],
                                         const uint4 (&hq0)[R], const uint4 (&hq1)[R], int g2,
                                         const XA &x, int e0, uint32_t one, uint32_t nib,
                                         float2 m1, float2 (&al)[R][NTOK][2],
                                         float2 (&ah)[R][NTOK][2]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float2 l01[R], l23[R], h01[R], h23[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t q = word_of(k < 4 ? w0[r] : w1[r], k % 4);
            const uint32_t hq = word_of(k < 4 ? hq0[r] : hq1[r], k % 4) >> g2;
            const uint32_t lo = bitsel(q, hq << 4, nib);
            const uint32_t hi = bitsel(q >> 4, hq << 3, nib);
            const uint32_t b3 = __byte_perm(lo, hi, 0x0703);  // lo byte 3 -> 0, hi byte 3 -> 2
            l01[r] = __fadd2_rn(f2(fone(lo, 0x1Fu, one), fone(lo, 0x1F00u, one)), m1);
            l23[r] = __fadd2_rn(f2(fone(lo, 0x1F0000u, one), fone(b3, 0x1Fu, one)), m1);
            h01[r] = __fadd2_rn(f2(fone(hi, 0x1Fu, one), fone(hi, 0x1F00u, one)), m1);
            h23[r] = __fadd2_rn(f2(fone(hi, 0x1F0000u, one), fone(b3, 0x1F0000u, one)), m1);
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t) {
            const float4 xl = x.xs4(t, e0 + 4 * k);
            const float4 xh = x.xs4(t, e0 + 32 + 4 * k);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                al[r][t][0] = __ffma2_rn(l01[r], make_float2(xl.x, xl.y), al[r][t][0]);
                al[r][t][1] = __ffma2_rn(l23[r], make_float2(xl.z, xl.w), al[r][t][1]);
                ah[r][t][0] = __ffma2_rn(h01[r], make_float2(xh.x, xh.y), ah[r][t][0]);
                ah[r][t][1] = __ffma2_rn(h23[r], make_float2(xh.z, xh.w), ah[r][t][1]);
            }
        }
    }
}

// Q4_K (Q5 = false; chunks: 0 header, 1..8 qs) and Q5_K (Q5 = true; 0
// header, 1..2 qh, 3..10 qs) for R rows of the same block column (B[r]).
// The four groups run as a loop (small code).  Each row's result is the
// same whatever R is.
template <int NTOK, bool Q5, int R, class BS, class XA>
__device__ __forceinline__ void block_q45(const BS (&B)[R], const XA &x, float (&part)[R][NTOK]) {
    const uint32_t one = reg_one();
    uint32_t nib, m23;
    asm("mov.b32 %0, 0x0F0F0F0F;" : "=r"(nib));
    asm("mov.b32 %0, 0x4B000000;" : "=r"(m23));
    const float2 m1 = make_float2(reg_f32(-1.0f), reg_f32(-1.0f));
    Q45Head hd[R];
    uint4 hq0[R], hq1[R];
    float acc[R][NTOK];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        hd[r] = Q45Head(B[r].v4(0));
        if (Q5) {
            hq0[r] = B[r].v4(1);
            hq1[r] = B[r].v4(2);
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t) acc[r][t] = 0.0f;
    }
    constexpr int QS = Q5 ? 3 : 1;
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
        float2 al[R][NTOK][2], ah[R][NTOK][2];
        uint4 w0[R], w1[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int t = 0; t < NTOK; ++t)
                al[r][t][0] = al[r][t][1] = ah[r][t][0] = ah[r][t][1] = make_float2(0.0f, 0.0f);
            w0[r] = B[r].v4(QS + 2 * g);
            w1[r] = B[r].v4(QS + 2 * g + 1);
        }
        if (Q5)
            q5_group<NTOK, R>(w0, w1, hq0, hq1, 2 * g, x, 64 * g, one, nib, m1, al, ah);
        else
            q4_group<NTOK, R>(w0, w1, x, 64 * g, one, m1, al, ah);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float2 ds = hd[r].scale_pair(g, m23);
#pragma unroll
            for (int t = 0; t < NTOK; ++t) {
                acc[r][t] = fmaf(ds.x, pair_sum(al[r][t][0], al[r][t][1]), acc[r][t]);
                acc[r][t] = fmaf(ds.y, pair_sum(ah[r][t][0], ah[r][t][1]), acc[r][t]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int t = 0; t < NTOK; ++t) part[r][t] = acc[r][t] - q45_min_term(hd[r], x, t, m23);
}

// ------------------------------------------------------------------ Q6_K
// A word source `W` returns block words (bytes 4k..4k+3 of the 210-byte
// block): W.words4(j, o) gives words j..j+3, W.dbits() the f16 d at bytes
// 208..209.  ql = words 0..31, qh = words 32..47, int8 scales = words 48..51.
// Half h (weights 128h..128h+127) reads ql bytes 64h.. and qh bytes 32h..;
// for l = 0..31 the weights 128h+l, +32, +64, +96 (quadrants 0..3) take the
// low nibble of ql[64h+l], the low nibble of ql[64h+32+l], the high nibble
// of ql[64h+l], the high nibble of ql[64h+32+l], and bit pairs 0-1, 2-3,
// 4-5, 6-7 of qh[32h+l].  Sub-block of weight e: e / 16 = 8h + 2*quadrant +
// k/4 for the word k = (e % 32) / 4.
template <int NTOK, class WS, class XA>
__device__ __forceinline__ void block_q6k(const WS &W, const XA &x, float (&part)[NTOK]) {
    const uint32_t one = reg_one();
    uint32_t nib, m23;
    asm("mov.b32 %0, 0x0F0F0F0F;" : "=r"(nib));
    asm("mov.b32 %0, 0x4B000000;" : "=r"(m23));
    // (code - 32) * 2^(o-23) = F - (1 + 32 * 2^(o-23)) for code bits at o
    const float2 c01 = make_float2(reg_f32(-(1.0f + 0x1p-18f)), reg_f32(-(1.0f + 0x1p-10f)));  // o = 0, 8
    const float2 c23e = make_float2(reg_f32(-(1.0f + 0x1p-2f)), reg_f32(-(1.0f + 0x1p-18f)));  // o = 16, 0
    const float2 c23o = make_float2(reg_f32(-(1.0f + 0x1p-2f)), reg_f32(-(1.0f + 0x1p-2f)));   // o = 16, 16
    const float d = h2f(W.dbits());
    uint32_t scw[4];
    W.words4(48, scw);
    // signed scale bytes biased to 0..255 for the magic-float decode
#pragma unroll
    for (int i = 0; i < 4; ++i) scw[i] ^= 0x80808080u;
    float acc[NTOK];
#pragma unroll
    for (int t = 0; t < NTOK; ++t) acc[t] = 0.0f;

    // iteration it: half h = it / 2 (weights 128h..), words k = 4kh..4kh+3
#pragma unroll 1
    for (int it = 0; it < 4; ++it) {
        const int h = it >> 1, kh = it & 1;
        uint32_t qa4[4], qb4[4], qh4[4];
        W.words4(16 * h + 4 * kh, qa4);
        W.words4(16 * h + 8 + 4 * kh, qb4);
        W.words4(32 + 8 * h + 4 * kh, qh4);
        const int e0 = 128 * h + 16 * kh;
        float2 a[NTOK][4][2];
#pragma unroll
        for (int t = 0; t < NTOK; ++t)
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) a[t][qd][0] = a[t][qd][1] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t qa = qa4[kk], qb = qb4[kk], qh = qh4[kk];
            uint32_t c[4];
            c[0] = bitsel(qa, qh << 4, nib);
            c[1] = bitsel(qb, qh << 2, nib);
            c[2] = bitsel(qa >> 4, qh, nib);
            c[3] = bitsel(qb >> 4, qh >> 2, nib);
            const uint32_t b01 = __byte_perm(c[0], c[1], 0x0703);  // c0.b3 -> 0, c1.b3 -> 2
            const uint32_t b23 = __byte_perm(c[2], c[3], 0x0703);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const uint32_t cw = c[qd];
                const uint32_t bp = qd < 2 ? b01 : b23;
                const uint32_t b3 = fone(bp, (qd & 1) ? 0x3F0000u : 0x3Fu, one);
                const float2 p01 = __fadd2_rn(f2(fone(cw, 0x3Fu, one), fone(cw, 0x3F00u, one)), c01);
                const float2 p23 = __fadd2_rn(f2(fone(cw, 0x3F0000u, one), b3), (qd & 1) ? c23o : c23e);
#pragma unroll
                for (int t = 0; t < NTOK; ++t) {
                    const float4 xv = x.xs4(t, e0 + 32 * qd + 4 * kk);
                    a[t][qd][0] = __ffma2_rn(p01, make_float2(xv.x, xv.y), a[t][qd][0]);
                    a[t][qd][1] = __ffma2_rn(p23, make_float2(xv.z, xv.w), a[t][qd][1]);
                }
            }
        }
        // scales of sub-blocks 8h + 2qd + kh (quadrants qd, qd + 1):
        // d * (F - (2^23 + 128)) with F = 2^23 + (sc + 128)
#pragma unroll
        for (int qd = 0; qd < 4; qd += 2) {
            const uint32_t w = h ? scw[2 + qd / 2] : scw[qd / 2];
            const float2 f = make_float2(__uint_as_float(__byte_perm(w, m23, 0x7650u | (uint32_t)kh)),
                                         __uint_as_float(__byte_perm(w, m23, 0x7650u | (2u + kh))));
            const float2 sc = __fmul2_rn(make_float2(d, d),
                                         __fadd2_rn(f, make_float2(-8388736.0f, -8388736.0f)));
#pragma unroll
            for (int t = 0; t < NTOK; ++t) {
                acc[t] = fmaf(sc.x, pair_sum(a[t][qd][0], a[t][qd][1]), acc[t]);
                acc[t] = fmaf(sc.y, pair_sum(a[t][qd + 1][0], a[t][qd + 1][1]), acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NTOK; ++t) part[t] = acc[t];
}

// Word sources for Q6_K blocks (2-byte aligned, so a block starts either 4-
// byte aligned or 2 bytes past a 4-byte boundary).
struct Q6GlobalAligned {
    const uint8_t *a;
    __device__ __forceinline__ void words4(int j, uint32_t (&o)[4]) const {
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = ldg_u32(a + 4 * (j + i));
    }
    __device__ __forceinline__ uint32_t dbits() const { return ldg_u16(a + 208); }
};
struct Q6GlobalShifted {  // a = block start - 2 (4-byte aligned)
    const uint8_t *a;
    __device__ __forceinline__ void words4(int j, uint32_t (&o)[4]) const {
        uint32_t r[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) r[i] = ldg_u32(a + 4 * (j + i));
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(r[i], r[i + 1], 16);
    }
    __device__ __forceinline__ uint32_t dbits() const { return ldg_u32(a + 208) >> 16; }
};

}  // namespace kq
