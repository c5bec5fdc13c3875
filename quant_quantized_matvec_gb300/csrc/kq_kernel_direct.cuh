// kq_kernel_direct.cuh -- the set kernel, direct-load variant.
//
// One CTA owns `rpc` consecutive rows of one member of the set.  Its
// (row, block) pairs are spread over the CTA's threads, block-column major,
// so neighbouring lanes take neighbouring rows of the same block column and
// read the same inputs.  Every thread loads its super-block straight from
// global memory with 16-byte (Q4_K, Q5_K) or 4-byte (Q6_K, whose 210-byte
// blocks are only 2-byte aligned) read-only loads, computes the block's
// contribution to each token (kq_blocks.cuh; inputs are read from global
// memory and scaled on the fly), and parks it in shared memory.
// After one barrier each (row, token) sums its blocks in block order 0..nb-1
// and writes y.  The sum order depends on nothing but nb, so a member's
// output is the same whichever set, grid or row split it runs in.
#pragma once

#include "kq_blocks.cuh"

namespace kq {

constexpr int kDirectThreads = 256;

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
        const float *xb = M.x + (int64_t)b * 256;
        float part[NTOK];
        if (M.fmt == kFmtQ4K) {
            const BlockGlobal B[1] = {{reinterpret_cast<const uint4 *>(M.W + blk_index * 144)}};
            float p1[1][NTOK];
            block_q45<NTOK, false, 1>(B, XGlobalS<true>{xb, cols}, p1);
#pragma unroll
            for (int t = 0; t < NTOK; ++t) part[t] = p1[0][t];
        } else if (M.fmt == kFmtQ5K) {
            const BlockGlobal B[1] = {{reinterpret_cast<const uint4 *>(M.W + blk_index * 176)}};
            float p1[1][NTOK];
            block_q45<NTOK, true, 1>(B, XGlobalS<false>{xb, cols}, p1);
#pragma unroll
            for (int t = 0; t < NTOK; ++t) part[t] = p1[0][t];
        } else {
            const uint8_t *a = M.W + blk_index * 210;
            if ((uintptr_t)a & 3u)
                block_q6k<NTOK>(Q6GlobalShifted{a - 2}, XGlobalS<false>{xb, cols}, part);
            else
                block_q6k<NTOK>(Q6GlobalAligned{a}, XGlobalS<false>{xb, cols}, part);
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
