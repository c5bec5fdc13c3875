// kq_tc.cuh -- one super-block column of 16 rows against 4..16 token
// columns on the tensor cores (m16n8k16, f16 operands, f32 accumulation),
// for Q4_K, Q5_K and Q6_K.
//
// Arithmetic ("Chapter 6 - The kquant family on the reference lane",
// sections 6.2 and 6.4; "Chapter 13 - The QKV + gate matvec family",
// section 13.4.2 for the deferred scaling).  With the inputs of kq_xtc.cuh
// (x_j ~ (hi_j + lo_j) * u per token and column) and the codes as f16
// (the f16 whose bits are an integer k < 2048 has the value k * 2^-24;
// Q6_K's codes become (q - 32) * 2^-24 by one exact f16 addition), an MMA
// chain over a sub-block gives
//
//   D = 2^-24 * sum_{j in sub-block} c_j * (hi_j + lo_j)
//
// for each (row, token), c = q (Q4_K, Q5_K) or q - 32 (Q6_K).  The chain is
// hi then lo for each k-step of 16 inputs (two k-steps per Q4_K / Q5_K
// sub-block of 32, one per Q6_K sub-block of 16).  Then, in this fixed
// order, per row and token of a block:
//
//   Q4_K / Q5_K   acc = 0; for s = 0..7:  acc = fma(F_s, D_s, acc),
//                 F_s = d * sc_s * 2^24 (exact);
//                 mt  = 0; for s = 0..7:  mt = fma(dm_s, S32_s, mt),
//                 dm_s = dmin * m_s (exact), S32 the sub-block input sums;
//                 v   = u * (acc - mt)
//   Q6_K          acc = 0; for h = 0, 1; kh = 0, 1; q = 0..3, i.e. sub-block
//                 s = 8h + 2q + kh in that order:  acc = fma(F_s, D_s, acc),
//                 F_s = d * sc_s * 2^24 (exact);  v = u * acc
//
// Every product of a code and an f16 term is exact; the tensor core's sums
// and these f32 steps round.  A zero Q6_K weight (q = 32) contributes
// exactly nothing.  A row's v depends only on its bytes and its token's
// inputs (each MMA output is one row against one token column), never on
// the tile, the other rows, the other tokens, the kernel or the launch.
//
// The k index inside a k-step is permuted (kq_xtc.cuh): lane t of a group
// of four takes inputs 4t, 4t + 2 (first A register of a row) and 4t + 1,
// 4t + 3 (second), i.e. bytes 0, 2 and 1, 3 of one 32-bit word of codes.
#pragma once

#include "kq_common.cuh"
#include "kq_xtc.cuh"

namespace kq {

// Per-warp scratch of a unit: 16 rows x kTcScrStride floats: F_0..F_15,
// then (Q4_K / Q5_K) dm_0..dm_7.  112-byte rows: a group of eight rows read
// together falls on eight different banks.
constexpr int kTcScrStride = 28;
constexpr int kTcScrBytes = 16 * kTcScrStride * 4;
// 16-row tiles of a streaming-kernel unit at most: with two octets of
// tokens a unit's input fragments are twice the bytes, and a group's two
// tiles (17..32 rows) share them; at one octet a unit is one tile (dealing
// twice as many units evens out the warps' work).  A consumer warp's
// scratch holds that many tiles' scales where the launch has such groups.
__host__ __device__ constexpr int tc_unit_tiles(int noct) { return noct >= 2 ? 2 : 1; }

// D += A * B over one 16 x 16 x 8 tile, f16 operands, f32 accumulators.
// (A pure register operation: not volatile, so loads may be scheduled
// across it.)
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (q - 32) * 2^-24 for both f16 halves of a (codes q * 2^-24, q < 64):
// exact, the result being a representable f16 (subnormals kept).
__device__ __forceinline__ uint32_t tc_minus32(uint32_t a) {
    uint32_t r;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(0x80208020u));
    return r;
}

template <bool GLOBAL, class T>
__device__ __forceinline__ T tc_ld(const void *p) {
    if (GLOBAL) return __ldg(reinterpret_cast<const T *>(p));
    return *reinterpret_cast<const T *>(p);
}

// Float 2^23 + byte k of w (a value below 256).
__device__ __forceinline__ float tc_magic_byte(uint32_t w, int k) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u | (uint32_t)k));
}

// A Q6_K block (2-byte aligned): word i (bytes 4i..4i+3) through aligned
// loads and a funnel shift.  Only a block that starts 2 bytes past a 4-byte
// boundary reads the aligned word after word i, which lies inside the
// block for every i < 52.
template <bool GLOBAL>
struct Q6Row {
    const uint8_t *a4;  // block start rounded down to 4 bytes
    uint32_t sh;        // 16 when the block starts 2 bytes past a 4-byte boundary
    static __device__ __forceinline__ Q6Row at(const uint8_t *p) {
        const uint32_t mis = (uint32_t)reinterpret_cast<uintptr_t>(p) & 3u;
        return {p - mis, mis * 8u};
    }
    __device__ __forceinline__ uint32_t word(int i) const {
        const uint32_t lo = tc_ld<GLOBAL, uint32_t>(a4 + 4 * i);
        const uint32_t hi = sh ? tc_ld<GLOBAL, uint32_t>(a4 + 4 * i + 4) : 0u;
        return __funnelshift_r(lo, hi, sh);
    }
    __device__ __forceinline__ uint32_t dbits() const {
        return sh ? (tc_ld<GLOBAL, uint32_t>(a4 + 208) >> 16)
                  : (uint32_t)tc_ld<GLOBAL, unsigned short>(a4 + 208);
    }
};

// The per-row scales of a unit into the warp's scratch: lane = row r (0..15)
// x half h.  Q4_K / Q5_K: F_s, dm_s for s = 4h..4h+3; Q6_K: F_s for
// s = 8h..8h+7.  `rowp(r)` is row r's block (rows past nvalid - 1 repeat
// row nvalid - 1).
template <int FMT, bool GW, class RowP>
__device__ __forceinline__ void tc_scales(RowP rowp, int nvalid, float *scr, int lane) {
    const int r = lane & 15, h = lane >> 4;
    const uint8_t *p = rowp(r < nvalid ? r : nvalid - 1);
    float *o = scr + r * kTcScrStride;
    if (FMT != kFmtQ6K) {
        const uint4 hd = tc_ld<GW, uint4>(p);
        const float d24 = h2f(hd.x) * 16777216.0f, nd24 = -d24 * 8388608.0f;
        const float dmin = h2f(hd.x >> 16), ndm = -dmin * 8388608.0f;
        const ScaleWords sw = unpack_scale_words(hd.y, hd.z, hd.w);
        const uint32_t scw = h ? sw.sc_hi : sw.sc_lo, mw = h ? sw.m_hi : sw.m_lo;
        float4 F, M;
        F.x = fmaf(d24, tc_magic_byte(scw, 0), nd24);
        F.y = fmaf(d24, tc_magic_byte(scw, 1), nd24);
        F.z = fmaf(d24, tc_magic_byte(scw, 2), nd24);
        F.w = fmaf(d24, tc_magic_byte(scw, 3), nd24);
        M.x = fmaf(dmin, tc_magic_byte(mw, 0), ndm);
        M.y = fmaf(dmin, tc_magic_byte(mw, 1), ndm);
        M.z = fmaf(dmin, tc_magic_byte(mw, 2), ndm);
        M.w = fmaf(dmin, tc_magic_byte(mw, 3), ndm);
        *reinterpret_cast<float4 *>(o + 4 * h) = F;
        *reinterpret_cast<float4 *>(o + 16 + 4 * h) = M;
    } else {
        const Q6Row<GW> q = Q6Row<GW>::at(p);
        const float d24 = h2f(q.dbits()) * 16777216.0f;
        // signed scale bytes biased to 0..255 for the magic-float decode:
        // d24 * (F - (2^23 + 128)) with F = 2^23 + (sc + 128)
        const uint32_t w0 = q.word(48 + 2 * h) ^ 0x80808080u;
        const uint32_t w1 = q.word(49 + 2 * h) ^ 0x80808080u;
        float4 F0, F1;
        F0.x = d24 * (tc_magic_byte(w0, 0) - 8388736.0f);
        F0.y = d24 * (tc_magic_byte(w0, 1) - 8388736.0f);
        F0.z = d24 * (tc_magic_byte(w0, 2) - 8388736.0f);
        F0.w = d24 * (tc_magic_byte(w0, 3) - 8388736.0f);
        F1.x = d24 * (tc_magic_byte(w1, 0) - 8388736.0f);
        F1.y = d24 * (tc_magic_byte(w1, 1) - 8388736.0f);
        F1.z = d24 * (tc_magic_byte(w1, 2) - 8388736.0f);
        F1.w = d24 * (tc_magic_byte(w1, 3) - 8388736.0f);
        *reinterpret_cast<float4 *>(o + 8 * h) = F0;
        *reinterpret_cast<float4 *>(o + 8 * h + 4) = F1;
    }
}

// A registers of one k-step from one word of code bytes per row (codes in
// the bytes' low bits, below 64): rows g (wa) and g + 8 (wb).
__device__ __forceinline__ void tc_a_from_bytes(uint32_t wa, uint32_t wb, uint32_t mask,
                                                uint32_t (&a)[4]) {
    a[0] = wa & mask;         // inputs 4t, 4t + 2 of row g
    a[1] = wb & mask;         // row g + 8
    a[2] = (wa >> 8) & mask;  // inputs 4t + 1, 4t + 3 of row g
    a[3] = (wb >> 8) & mask;
}

// One unit: MT tiles of 16 rows (tile m = rows 16m..16m+15 at rowp(r); rows
// past nvalid - 1 repeat row nvalid - 1), one block column, NOCT octets of
// tokens; `col` = this column's input records (kq_xtc.cuh: the fragments of
// octets 0..NOCT-1, then the aux of tokens 0..8 NOCT - 1), in global memory
// (GB) or shared memory; `ntok` the launch's token columns.  GW: the weights
// are in global memory.  The tiles share every B fragment load; each tile's
// operations are those of a one-tile unit, in the same order.  `scr` holds
// MT tiles' scales (MT x kTcScrBytes).  Returns v[m][o][k2][j] for row
// 16m + g + 8 k2 and token 8o + 2t + j in lane (g, t); tokens past ntok are
// garbage and not to be stored.
template <int FMT, int NOCT, bool GW, bool GB, int MT, class RowP>
__device__ __forceinline__ void tc_unit_mt(RowP rowp, int nvalid, const uint8_t *col, int ntok,
                                           float *scr, int lane, float (&v)[MT][NOCT][2][2]) {
    const uint8_t *frag = col;
    constexpr int ostride = kTcFragOctBytes;
    const float *aux = reinterpret_cast<const float *>(col + NOCT * kTcFragOctBytes);
    constexpr int taux = kTcAuxFloats;
    // One octet from global memory: all 16 k-steps' B fragments are
    // requested before anything else, so that the unit waits on L2 once
    // rather than once per sub-block.
    constexpr bool PRE = GB && NOCT == 1;
    uint4 bpre[PRE ? 16 : 1];
    if constexpr (PRE) {
#pragma unroll
        for (int k = 0; k < 16; ++k) bpre[k] = tc_ld<true, uint4>(col + tc_frag_offset(k, lane));
    }
    auto bfrag = [&](const uint8_t *fo, int k) -> uint4 {
        if constexpr (PRE) return bpre[k];
        return tc_ld<GB, uint4>(fo + tc_frag_offset(k, 0));
    };
#pragma unroll
    for (int m = 0; m < MT; ++m)
        tc_scales<FMT, GW>([&](int r) { return rowp(16 * m + r); }, nvalid - 16 * m,
                           scr + 16 * m * kTcScrStride, lane);
    __syncwarp();
    const int g = lane >> 2, t = lane & 3;
    const uint8_t *pa[MT], *pb[MT];
    const float *Fa[MT], *Fb[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int ra = 16 * m + g, rb = ra + 8;
        pa[m] = rowp(ra < nvalid ? ra : nvalid - 1);
        pb[m] = rowp(rb < nvalid ? rb : nvalid - 1);
        Fa[m] = scr + ra * kTcScrStride;
        Fb[m] = scr + rb * kTcScrStride;
    }
    float acc[MT][NOCT][2][2];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int o = 0; o < NOCT; ++o)
            acc[m][o][0][0] = acc[m][o][0][1] = acc[m][o][1][0] = acc[m][o][1][1] = 0.0f;
    const uint8_t *fl = frag + lane * 16;
    if (FMT != kFmtQ6K) {
        constexpr bool Q5 = FMT == kFmtQ5K;
        constexpr int QS = Q5 ? 48 : 16;
        const uint32_t m4 = 0x000F000Fu, m5 = 0x001F001Fu;
        uint32_t qha[MT][2], qhb[MT][2];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            qha[m][0] = qha[m][1] = qhb[m][0] = qhb[m][1] = 0u;
            if (Q5) {  // qh bytes 16 * half + 4t .. + 3 of the two rows
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    qha[m][hf] = tc_ld<GW, uint32_t>(pa[m] + 16 + 16 * hf + 4 * t);
                    qhb[m][hf] = tc_ld<GW, uint32_t>(pb[m] + 16 + 16 * hf + 4 * t);
                }
            }
        }
#pragma unroll
        for (int gp = 0; gp < 4; ++gp) {
            // qs words of k-step halves 0 and 1 of group gp (sub-blocks 2gp, 2gp + 1)
            uint32_t wa[MT][2], wb[MT][2];
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    wa[m][hf] = tc_ld<GW, uint32_t>(pa[m] + QS + 32 * gp + 16 * hf + 4 * t);
                    wb[m][hf] = tc_ld<GW, uint32_t>(pb[m] + QS + 32 * gp + 16 * hf + 4 * t);
                }
            // one octet: the two sub-blocks' scales of row g in one 8-byte
            // load (row g + 8's too spilled registers and slowed the Q6_K
            // path of the same kernel; at two octets, scalar loads)
            float2 fa2[MT];
            if constexpr (NOCT == 1) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    fa2[m] = *reinterpret_cast<const float2 *>(Fa[m] + 2 * gp);
            }
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
                const int s = 2 * gp + hi;
                uint32_t A[MT][2][4];
                float fa[MT], fb[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t ca = hi ? (wa[m][hf] >> 4) & 0x0F0F0F0Fu : wa[m][hf] & 0x0F0F0F0Fu;
                        uint32_t cb = hi ? (wb[m][hf] >> 4) & 0x0F0F0F0Fu : wb[m][hf] & 0x0F0F0F0Fu;
                        if (Q5) {  // bit s of each qh byte as bit 4 of the code
                            ca |= (s <= 4 ? qha[m][hf] << (4 - s) : qha[m][hf] >> (s - 4)) & 0x10101010u;
                            cb |= (s <= 4 ? qhb[m][hf] << (4 - s) : qhb[m][hf] >> (s - 4)) & 0x10101010u;
                        }
                        tc_a_from_bytes(ca, cb, Q5 ? m5 : m4, A[m][hf]);
                    }
                    if constexpr (NOCT == 1) {
                        fa[m] = hi ? fa2[m].y : fa2[m].x;
                        fb[m] = Fb[m][s];
                    } else {
                        fa[m] = Fa[m][s];
                        fb[m] = Fb[m][s];
                    }
                }
#pragma unroll
                for (int o = 0; o < NOCT; ++o) {
                    const uint8_t *fo = fl + o * ostride;
                    float D[MT][4];
#pragma unroll
                    for (int m = 0; m < MT; ++m) D[m][0] = D[m][1] = D[m][2] = D[m][3] = 0.0f;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const uint4 b = bfrag(fo, 2 * s + hf);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            mma_f16(D[m], A[m][hf], b.x, b.y);  // hi
                            mma_f16(D[m], A[m][hf], b.z, b.w);  // lo
                        }
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        acc[m][o][0][0] = fmaf(fa[m], D[m][0], acc[m][o][0][0]);
                        acc[m][o][0][1] = fmaf(fa[m], D[m][1], acc[m][o][0][1]);
                        acc[m][o][1][0] = fmaf(fb[m], D[m][2], acc[m][o][1][0]);
                        acc[m][o][1][1] = fmaf(fb[m], D[m][3], acc[m][o][1][1]);
                    }
                }
            }
        }
        // v = u * (acc - mt), mt = fma chain of dm_s * S32_s over s
#pragma unroll
        for (int o = 0; o < NOCT; ++o) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                int tok = 8 * o + 2 * t + j;
                tok = tok < ntok ? tok : ntok - 1;
                const float *ax = aux + tok * taux;
                const float4 s0 = tc_ld<GB, float4>(ax + kTcAuxS32);
                const float4 s1 = tc_ld<GB, float4>(ax + kTcAuxS32 + 4);
                const float u = tc_ld<GB, float>(ax + kTcAuxU);
                const float S[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        // dm_0..dm_7 of the row (one octet: 16-byte loads)
                        const float *dp = (k2 ? Fb[m] : Fa[m]) + 16;
                        float dm[8];
                        if constexpr (NOCT == 1) {
                            const float4 d0 = *reinterpret_cast<const float4 *>(dp);
                            const float4 d1 = *reinterpret_cast<const float4 *>(dp + 4);
                            dm[0] = d0.x; dm[1] = d0.y; dm[2] = d0.z; dm[3] = d0.w;
                            dm[4] = d1.x; dm[5] = d1.y; dm[6] = d1.z; dm[7] = d1.w;
                        } else {
#pragma unroll
                            for (int q = 0; q < 8; ++q) dm[q] = dp[q];
                        }
                        float mt = dm[0] * S[0];
#pragma unroll
                        for (int s = 1; s < 8; ++s) mt = fmaf(dm[s], S[s], mt);
                        v[m][o][k2][j] = u * (acc[m][o][k2][j] - mt);
                    }
            }
        }
    } else {
        const uint32_t m6 = 0x003F003Fu;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {
                // ql words (quadrant pairs 0/2 and 1/3) and the qh word of
                // inputs 128h + 16kh + 4t .. (+32q) of the two rows
                const int w0 = 16 * h + 4 * kh + t, w1 = w0 + 8, wq = 32 + 8 * h + 4 * kh + t;
                uint32_t la0[MT], la1[MT], lqa[MT], lb0[MT], lb1[MT], lqb[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const Q6Row<GW> qa = Q6Row<GW>::at(pa[m]), qb = Q6Row<GW>::at(pb[m]);
                    la0[m] = qa.word(w0);
                    la1[m] = qa.word(w1);
                    lqa[m] = qa.word(wq);
                    lb0[m] = qb.word(w0);
                    lb1[m] = qb.word(w1);
                    lqb[m] = qb.word(wq);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int s = 8 * h + 2 * q + kh;
                    uint32_t A[MT][4];
                    float fa[MT], fb[MT];
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint32_t la = (q & 1) ? la1[m] : la0[m], lb = (q & 1) ? lb1[m] : lb0[m];
                        const uint32_t ca = (q < 2 ? la & 0x0F0F0F0Fu : (la >> 4) & 0x0F0F0F0Fu) |
                                            (((lqa[m] >> (2 * q)) & 0x03030303u) << 4);
                        const uint32_t cb = (q < 2 ? lb & 0x0F0F0F0Fu : (lb >> 4) & 0x0F0F0F0Fu) |
                                            (((lqb[m] >> (2 * q)) & 0x03030303u) << 4);
                        tc_a_from_bytes(ca, cb, m6, A[m]);
#pragma unroll
                        for (int i = 0; i < 4; ++i) A[m][i] = tc_minus32(A[m][i]);
                        fa[m] = Fa[m][s];
                        fb[m] = Fb[m][s];
                    }
#pragma unroll
                    for (int o = 0; o < NOCT; ++o) {
                        const uint8_t *fo = fl + o * ostride;
                        const uint4 b = bfrag(fo, s);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            mma_f16(D, A[m], b.x, b.y);  // hi
                            mma_f16(D, A[m], b.z, b.w);  // lo
                            acc[m][o][0][0] = fmaf(fa[m], D[0], acc[m][o][0][0]);
                            acc[m][o][0][1] = fmaf(fa[m], D[1], acc[m][o][0][1]);
                            acc[m][o][1][0] = fmaf(fb[m], D[2], acc[m][o][1][0]);
                            acc[m][o][1][1] = fmaf(fb[m], D[3], acc[m][o][1][1]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int o = 0; o < NOCT; ++o) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                int tok = 8 * o + 2 * t + j;
                tok = tok < ntok ? tok : ntok - 1;
                const float u = tc_ld<GB, float>(aux + tok * taux + kTcAuxU);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    v[m][o][0][j] = u * acc[m][o][0][j];
                    v[m][o][1][j] = u * acc[m][o][1][j];
                }
            }
        }
    }
    __syncwarp();  // the scratch is free for the next unit
}

// One tile of 16 rows (tc_unit_mt with MT = 1): v[o][k2][j] for row g + 8 k2.
template <int FMT, int NOCT, bool GW, bool GB, class RowP>
__device__ __forceinline__ void tc_unit(RowP rowp, int nvalid, const uint8_t *col, int ntok,
                                        float *scr, int lane, float (&v)[NOCT][2][2]) {
    tc_unit_mt<FMT, NOCT, GW, GB, 1>(rowp, nvalid, col, ntok, scr, lane,
                                     *reinterpret_cast<float (*)[1][NOCT][2][2]>(&v));
}

}  // namespace kq
