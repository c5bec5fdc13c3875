// kq_kernel_direct.cuh -- the set kernel, direct-load variant, and the pass
// that writes the input records to global memory for it.
//
// One CTA owns `rpc` consecutive rows of one member of the set.  Its
// (row, block) pairs are spread over the CTA's threads, block-column major,
// so neighbouring lanes take neighbouring rows of the same block column and
// read the same input record.  Every thread loads its super-block straight
// from global memory with 16-byte (Q4_K, Q5_K) or 4-byte (Q6_K, whose
// 210-byte blocks are only 2-byte aligned) read-only loads, computes the
// block's contribution to each token (kq_blocks.cuh, one row at a time)
// from the records in global memory, and parks it in shared memory.  After
// one barrier each (row, token) sums its blocks in block order 0..nb-1 and
// writes y.  The sum order depends on nothing but nb, so a member's output
// is the same whichever set, grid or row split it runs in, and the same as
// the streaming kernel's.
#pragma once

#include "kq_blocks.cuh"
#include "kq_tc.cuh"

namespace kq {

constexpr int kDirectThreads = 256;
constexpr int kPrepThreads = 256;

// Input records in global memory for each member (kq_xprep in kq_api.cu):
// warp w of the grid builds one 128-input half (kq_xrec.cuh).  Members are
// laid out one after another in warp order (first_warp).
struct PrepParams {
    const float *x[kMaxSet];
    uint8_t *rec[kMaxSet];
    int32_t nb[kMaxSet];
    int32_t q6[kMaxSet];
    int64_t first_warp[kMaxSet + 1];
    int32_t n;
    int32_t ntok;
};

constexpr int kDirectWarps = kDirectThreads / 32;

// Dynamic shared memory of the direct kernel for a member of rpc rows: the
// partials [nb][rpc][NTOK], then, for tensor-core launches, one unit
// scratch per warp.
__host__ __device__ constexpr int64_t direct_part_floats(int nb, int rpc, int ntok) {
    return ((int64_t)nb * rpc * ntok + 3) / 4 * 4;
}
__host__ __device__ constexpr int64_t direct_smem_bytes(int nb, int rpc, int ntok, bool tc) {
    return 4 * direct_part_floats(nb, rpc, ntok) + (tc ? kDirectWarps * kTcScrBytes : 0);
}

// The tensor-core form of a CTA: its rows cut into 16-row tiles, each warp
// taking (tile, block column) units in turn (kq_tc.cuh), weights and input
// fragments read from global memory.
template <int NOCT>
__device__ __forceinline__ void direct_tc(const SetParams &p, const MatDesc &M, int64_t r0,
                                          int R, float *part_s) {
    constexpr int NT = 8 * NOCT;
    const int nb = M.nb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *scr = part_s + direct_part_floats(nb, M.rpc, NT) + warp * (kTcScrBytes / 4);
    const int bb = M.fmt == kFmtQ4K ? 144 : M.fmt == kFmtQ5K ? 176 : 210;
    const int64_t rs = (int64_t)nb * bb;
    constexpr int colb = tc_col_bytes(NOCT);
    const int tiles = (R + 15) >> 4;
#pragma unroll 1
    for (int u = warp; u < tiles * nb; u += kDirectWarps) {
        const int b = u / tiles, tile = u - b * tiles;
        const int rt = tile * 16;
        const int nvalid = R - rt < 16 ? R - rt : 16;
        const uint8_t *blk = M.W + (r0 + rt) * rs + (int64_t)b * bb;
        const uint8_t *col = M.rec + (int64_t)b * colb;  // this column's records
        auto rowp = [&](int r) { return blk + r * rs; };
        float v[NOCT][2][2];
        if (M.fmt == kFmtQ4K)
            tc_unit<kFmtQ4K, NOCT, true, true>(rowp, nvalid, col, p.ntok, scr, lane, v);
        else if (M.fmt == kFmtQ5K)
            tc_unit<kFmtQ5K, NOCT, true, true>(rowp, nvalid, col, p.ntok, scr, lane, v);
        else
            tc_unit<kFmtQ6K, NOCT, true, true>(rowp, nvalid, col, p.ntok, scr, lane, v);
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            const int r = rt + g + 8 * k2;
            if (r < R) {
#pragma unroll
                for (int o = 0; o < NOCT; ++o)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        part_s[(b * R + r) * NT + 8 * o + 2 * t4 + j] = v[o][k2][j];
            }
        }
    }
}

template <int NTOK, bool TC>
__global__ void __launch_bounds__(kDirectThreads)
    kq_set_direct(const __grid_constant__ SetParams p) {
    extern __shared__ __align__(16) float part_s[];  // [nb][R][NTOK], then scratch

    int mi = 0;
#pragma unroll 1
    for (int i = 1; i < p.n; ++i)
        if ((int)blockIdx.x >= p.m[i].cta_begin) mi = i;
    const MatDesc &M = p.m[mi];
    const int64_t r0 = (int64_t)((int)blockIdx.x - M.cta_begin) * M.rpc;
    const int R = (int)min((int64_t)M.rpc, M.rows - r0);
    const int nb = M.nb;
    if constexpr (TC) {
        direct_tc<NTOK / 8>(p, M, r0, R, part_s);
    } else {
    const int tasks = R * nb;
#pragma unroll 1
    for (int task = threadIdx.x; task < tasks; task += kDirectThreads) {
        const int b = task / R;
        const int r = task - b * R;
        const int64_t blk_index = (r0 + r) * nb + b;
        float part[1][NTOK];
        if (M.fmt == kFmtQ6K) {
            const Rec<true> xr{M.rec + (int64_t)b * kRecQ6, nb * kRecQ6};
            const uint8_t *a = M.W + blk_index * 210;
            if ((uintptr_t)a & 3u) {
                const Q6Words<true, true> W[1] = {{a - 2}};
                block_q6k<NTOK, 1>(W, xr, part);
            } else {
                const Q6Words<false, true> W[1] = {{a}};
                block_q6k<NTOK, 1>(W, xr, part);
            }
        } else {
            const Rec<true> xr{M.rec + (int64_t)b * kRecQ45, nb * kRecQ45};
            if (M.fmt == kFmtQ4K) {
                const BlockGlobal B[1] = {{reinterpret_cast<const uint4 *>(M.W + blk_index * 144)}};
                block_q45<NTOK, false, 1>(B, xr, part);
            } else {
                const BlockGlobal B[1] = {{reinterpret_cast<const uint4 *>(M.W + blk_index * 176)}};
                block_q45<NTOK, true, 1>(B, xr, part);
            }
        }
#pragma unroll
        for (int t = 0; t < NTOK; ++t) part_s[(b * R + r) * NTOK + t] = part[0][t];
    }
    }
    __syncthreads();

#pragma unroll 1
    for (int o = threadIdx.x; o < R * NTOK; o += kDirectThreads) {
        const int r = o / NTOK, t = o - (o / NTOK) * NTOK;
        if (TC && t >= p.ntok) continue;
        float s = part_s[r * NTOK + t];
#pragma unroll 1
        for (int b = 1; b < nb; ++b) s += part_s[(b * R + r) * NTOK + t];
        M.y[(int64_t)t * M.rows + r0 + r] = s;
    }
}

}  // namespace kq
