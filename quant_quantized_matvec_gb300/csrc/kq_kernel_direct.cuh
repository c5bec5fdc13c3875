// kq_kernel_direct.cuh -- the set kernel, direct-load variant.
//
// One CTA owns `rpc` consecutive rows of one member of the set.  Its
// (row, block) pairs are spread over the CTA's threads, block-column major,
// so neighbouring lanes take neighbouring rows of the same block column and
// read the same inputs.  Every thread loads its super-block straight from
// global memory with 16-byte (Q4_K, Q5_K) or 4-byte (Q6_K, whose 210-byte
// blocks are only 2-byte aligned) read-only loads, computes the block's
// contribution to each token (kq_blocks.cuh), and parks it in shared memory.
// After one barrier each (row, token) sums its blocks in block order 0..nb-1
// and writes y.  The sum order depends on nothing but nb, so a member's
// output is the same whichever set, grid or row split it runs in.
#pragma once

#include "kq_blocks.cuh"

namespace kq {

constexpr int kDirectThreads = 256;

// Load one Q6_K block at byte address a (2-byte aligned) as 52 words of
// block bytes 4k..4k+3 plus the f16 d, without touching bytes outside the
// block except the two before it when a is 2 mod 4 (they belong to the
// previous block of the same matrix, which exists because the matrix start
// is 16-byte aligned).
__device__ __forceinline__ void load_q6(const uint8_t *a, uint32_t (&L)[52],
                                        uint32_t &dbits) {
    const uint32_t mis = (uint32_t)((uintptr_t)a & 3u);  // 0 or 2
    const uint8_t *base = a - mis;
    const uint32_t s = mis * 8u;
    uint32_t raw[53];
#pragma unroll
    for (int k = 0; k < 52; ++k) raw[k] = ldg_u32(base + 4 * k);
    raw[52] = mis ? ldg_u32(base + 208) : ldg_u16(base + 208);
#pragma unroll
    for (int k = 0; k < 52; ++k) L[k] = __funnelshift_r(raw[k], raw[k + 1], s);
    dbits = (raw[52] >> s) & 0xFFFFu;
}

template <int NTOK>
__global__ void __launch_bounds__(kDirectThreads)
    kq_set_direct(const __grid_constant__ SetParams p) {
    extern __shared__ float part_s[];  // [nb][R][NTOK]

    int mi = 0;
#pragma unroll 1
    for (int i = 1; i < p.n; ++i)
        if ((int)blockIdx.x >= p.m[i].cta_begin) mi = i;
    const MatDesc &M = p.m[mi];
    const int64_t r0 = (int64_t)((int)blockIdx.x - M.cta_begin) * M.rpc;
    const int R = (int)min((int64_t)M.rpc, M.rows - r0);
    const int nb = M.nb;
    const int64_t cols = (int64_t)nb * 256;
    const int tasks = R * nb;

#pragma unroll 1
    for (int task = threadIdx.x; task < tasks; task += kDirectThreads) {
        const int b = task / R;
        const int r = task - b * R;
        const int64_t blk_index = (r0 + r) * nb + b;
        const XGlobal xb{M.x + (int64_t)b * 256, cols};
        float part[NTOK];
        if (M.fmt == kFmtQ4K) {
            const uint8_t *a = M.W + blk_index * 144;
            uint4 v[9];
#pragma unroll
            for (int i = 0; i < 9; ++i) v[i] = ldg_v4(a + 16 * i);
            block_q45<NTOK, false>(v, xb, part);
        } else if (M.fmt == kFmtQ5K) {
            const uint8_t *a = M.W + blk_index * 176;
            uint4 v[11];
#pragma unroll
            for (int i = 0; i < 11; ++i) v[i] = ldg_v4(a + 16 * i);
            block_q45<NTOK, true>(v, xb, part);
        } else {
            uint32_t L[52], dbits;
            load_q6(M.W + blk_index * 210, L, dbits);
            block_q6<NTOK>(L, dbits, xb, part);
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t) part_s[(b * R + r) * NTOK + t] = part[t];
    }
    __syncthreads();

#pragma unroll 1
    for (int o = threadIdx.x; o < R * NTOK; o += kDirectThreads) {
        const int r = o / NTOK, t = o - (o / NTOK) * NTOK;
        float s = part_s[r * NTOK + t];
#pragma unroll 1
        for (int b = 1; b < nb; ++b) s += part_s[(b * R + r) * NTOK + t];
        M.y[(int64_t)t * M.rows + r0 + r] = s;
    }
}

}  // namespace kq
