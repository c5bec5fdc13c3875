// kq_kernel_stream.cuh -- the set kernel, TMA-streaming variant.
//
// One CTA per SM.  Each CTA owns a balanced, contiguous row range of one
// member of the set, split into row groups of at most 32 rows (Q4_K, Q5_K)
// or 16 rows (Q6_K).  A producer warp streams the weights through a ring of
// shared-memory slots:
//   * Q4_K / Q5_K: one 2-D tensor-map box per stage, [h rows][kb blocks]
//     (kb = 7: 1008 B / 1232 B per row, an odd number of 16-byte units, so
//     rows land on distinct shared-memory banks), cp.async.bulk.tensor;
//   * Q6_K: the group's whole rows, which are contiguous in memory but only
//     2-byte aligned, as 16-byte-aligned bulk copies (cp.async.bulk) of at
//     most 32 KiB, the sub-16-byte tail at the end of the matrix copied by
//     the producer with plain loads.
// Every consumer warp takes part in every stage: the stage's (row, block)
// pairs, ordered block-major so neighbouring lanes share inputs, are dealt
// out 32 at a time round-robin over the consumer warps, and each lane turns
// one super-block into per-token partial sums (kq_blocks.cuh) stored in
// shared memory.  When a row group's last stage is done the consumers sum
// each row's blocks in block order 0..nb-1 and write y.  That sum order, and
// each block's arithmetic, depend only on the format, nb and ntok, so a
// member's output is independent of the grid, the row split and the set.
//
// Waits on mbarriers are bounded by wall time.  A wait that expires sets
// the CTA's abort flag and the device error word; from then on no thread
// waits again, every named barrier is still reached, and the CTA's outputs
// are set to NaN, so a failure is reported instead of hanging the GPU.
#pragma once

#include <cuda.h>

#include "kq_blocks.cuh"

namespace kq {

constexpr int kStreamConsumers = 8;
constexpr int kStreamThreads = 32 * (kStreamConsumers + 1);
constexpr int kMaxMaps = 4;
constexpr int kMaxSlots = 32;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

struct StreamMember {
    const uint8_t *W;
    const float *x;
    float *y;
    int64_t rows;
    int32_t nb;
    int32_t fmt;
    int32_t cta_begin;
    int32_t ncta;
    int32_t rmax;   // rows per group at most
    int32_t kb;     // blocks per box (Q4_K / Q5_K)
    int32_t nmaps;  // tensor maps (box heights) for this member
    int32_t map_h[kMaxMaps];
};

struct StreamParams {
    CUtensorMap maps[kMaxSet][kMaxMaps];
    StreamMember m[kMaxSet];
    int32_t n;
    int32_t nslot;
    int32_t slot_bytes;
    int32_t x_bytes;     // 0: inputs are read from global memory
    int32_t part_bytes;
    unsigned int *err;   // device error word (nonzero: a wait expired)
};

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `parity` to complete; false once the wall-time limit
// passes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src,
                                         uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes"
        " [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tensor2d_g2s(uint32_t dst, const CUtensorMap *map,
                                             int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(kStreamConsumers * 32) : "memory");
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// A Q6_K block at shared address a (2-byte aligned) as 52 words + d.  Reads
// the two bytes before the block when a is 2 mod 4 and the two after it
// otherwise; both stay inside the stage's slot.
__device__ __forceinline__ void lds_q6(uint32_t a, uint32_t (&L)[52],
                                       uint32_t &dbits) {
    const uint32_t mis = a & 3u;
    const uint32_t base = a - mis;
    const uint32_t s = mis * 8u;
    uint32_t raw[53];
#pragma unroll
    for (int k = 0; k < 53; ++k) raw[k] = lds_u32(base + 4 * k);
#pragma unroll
    for (int k = 0; k < 52; ++k) L[k] = __funnelshift_r(raw[k], raw[k + 1], s);
    dbits = (raw[52] >> s) & 0xFFFFu;
}

// Row-group geometry of a CTA: rows [ra, ra + n) split into ng groups.
struct Groups {
    int64_t ra;
    int n, ng;
    __device__ __forceinline__ int64_t start(int g) const {
        return ra + (int64_t)g * n / ng;
    }
};

template <int NTOK, bool XSMEM>
__global__ void __launch_bounds__(kStreamThreads, 1)
    kq_set_stream(const __grid_constant__ StreamParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int abort_flag;

    int mi = 0;
#pragma unroll 1
    for (int i = 1; i < p.n; ++i)
        if ((int)blockIdx.x >= p.m[i].cta_begin) mi = i;
    const StreamMember &M = p.m[mi];
    const int fmt = M.fmt;
    const int nb = M.nb;
    const int bb = fmt == kFmtQ4K ? 144 : fmt == kFmtQ5K ? 176 : 210;
    const int64_t row_bytes = (int64_t)nb * bb;
    const int cidx = (int)blockIdx.x - M.cta_begin;
    Groups G;
    G.ra = M.rows * cidx / M.ncta;
    G.n = (int)(M.rows * (cidx + 1) / M.ncta - G.ra);
    G.ng = (G.n + M.rmax - 1) / M.rmax;
    const bool q6 = fmt == kFmtQ6K;
    const int nbox = q6 ? 1 : (nb + M.kb - 1) / M.kb;
    const int nstage = G.ng * nbox;
    const int nslot = p.nslot;

    const uint32_t bars = smem_addr(smem);  // full[0..nslot), empty[..]
    const uint32_t xs = bars + 1024;
    const uint32_t parts = xs + p.x_bytes;
    const uint32_t ring = parts + p.part_bytes;
    float *part_f = reinterpret_cast<float *>(smem + 1024 + p.x_bytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < nslot; ++s) {
            mbar_init(bars + 8 * s, 1);
            mbar_init(bars + 8 * (kMaxSlots + s), kStreamConsumers);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kStreamConsumers) {
        // ------------------------------------------------ producer
        if (lane != 0) return;
        int issued = 0;
        for (int s = 0; s < nstage; ++s) {
            const int slot = s % nslot;
            if (s >= nslot) {
                if (*(volatile int *)&abort_flag) break;
                if (!mbar_wait(bars + 8 * (kMaxSlots + slot), ((s / nslot) - 1) & 1)) {
                    atomicExch(&abort_flag, 1);
                    atomicOr(p.err, 1u);
                    break;
                }
            }
            const int g = s / nbox, k = s - (s / nbox) * nbox;
            const int64_t g0 = G.start(g), g1 = G.start(g + 1);
            const int h = (int)(g1 - g0);
            const uint32_t dst = ring + (uint32_t)slot * p.slot_bytes;
            const uint32_t full = bars + 8 * slot;
            if (!q6) {
                int mj = 0;
                for (int j = 0; j < M.nmaps; ++j)
                    if (M.map_h[j] == h) mj = j;
                const int box_row = M.kb * bb;
                mbar_expect_tx(full, (uint32_t)(h * box_row));
                tensor2d_g2s(dst, &p.maps[mi][mj], k * (box_row / 8), (int)g0, full);
            } else {
                const int64_t total = M.rows * row_bytes;
                const int64_t A = g0 * row_bytes, B = g1 * row_bytes;
                const int64_t A16 = A & ~(int64_t)15;
                int64_t B16 = (B + 15) & ~(int64_t)15;
                if (B16 > total) B16 = total & ~(int64_t)15;
                // sub-16-byte tail at the very end of the matrix
                uint8_t *dstp = smem + (dst - bars);
                for (int64_t i = B16; i < B; ++i) dstp[i - A16] = M.W[i];
                mbar_expect_tx(full, (uint32_t)(B16 - A16));
                for (int64_t o = A16; o < B16; o += 32768) {
                    const int64_t len = (B16 - o) < 32768 ? (B16 - o) : 32768;
                    bulk_g2s(dst + (uint32_t)(o - A16), M.W + o, (uint32_t)len, full);
                }
            }
            issued = s + 1;
        }
        if (*(volatile int *)&abort_flag) {
            // do not leave copies in flight into this CTA's shared memory
            for (int slot = 0; slot < nslot && slot < issued; ++slot) {
                const int last = slot + ((issued - 1 - slot) / nslot) * nslot;
                mbar_wait(bars + 8 * slot, (last / nslot) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int64_t cols = (int64_t)nb * 256;
    if (XSMEM) {
        const float4 *src = reinterpret_cast<const float4 *>(M.x);
        float4 *dstx = reinterpret_cast<float4 *>(smem + 1024);
        const int n4 = (int)(NTOK * cols / 4);
        for (int i = threadIdx.x; i < n4; i += kStreamConsumers * 32) dstx[i] = __ldg(src + i);
    }
    consumer_sync();

    int batch_base = 0;
#pragma unroll 1
    for (int s = 0; s < nstage; ++s) {
        const int slot = s % nslot;
        const int g = s / nbox, k = s - (s / nbox) * nbox;
        const int64_t g0 = G.start(g), g1 = G.start(g + 1);
        const int h = (int)(g1 - g0);
        const int b0 = q6 ? 0 : k * M.kb;
        const int kbv = q6 ? nb : (nb - b0 < M.kb ? nb - b0 : M.kb);
        const int tasks = h * kbv;
        const int nbat = (tasks + 31) / 32;
        const uint32_t sdata = ring + (uint32_t)slot * p.slot_bytes;
        bool ok = !*(volatile int *)&abort_flag;
        if (ok && !mbar_wait(bars + 8 * slot, (s / nslot) & 1)) {
            atomicExch(&abort_flag, 1);
            atomicOr(p.err, 1u);
            ok = false;
        }
        if (ok) {
            // stage-local byte offset of row r, block j
            const uint32_t q6off = q6 ? (uint32_t)((g0 * row_bytes) & 15) : 0u;
            int bat = batch_base + ((warp - batch_base % kStreamConsumers) + kStreamConsumers) %
                                       kStreamConsumers;
#pragma unroll 1
            for (; bat < batch_base + nbat; bat += kStreamConsumers) {
                const int t = (bat - batch_base) * 32 + lane;
                if (t >= tasks) continue;
                const int j = t / h, r = t - (t / h) * h;
                const int b = b0 + j;
                float part[NTOK];
                if (XSMEM) {
                    const XShared xa{xs + (uint32_t)(b * 1024), (uint32_t)(cols * 4)};
                    if (fmt == kFmtQ4K) {
                        uint4 v[9];
                        const uint32_t a = sdata + (uint32_t)(r * M.kb * 144 + j * 144);
#pragma unroll
                        for (int i = 0; i < 9; ++i) v[i] = lds_v4(a + 16 * i);
                        block_q45<NTOK, false>(v, xa, part);
                    } else if (fmt == kFmtQ5K) {
                        uint4 v[11];
                        const uint32_t a = sdata + (uint32_t)(r * M.kb * 176 + j * 176);
#pragma unroll
                        for (int i = 0; i < 11; ++i) v[i] = lds_v4(a + 16 * i);
                        block_q45<NTOK, true>(v, xa, part);
                    } else {
                        uint32_t L[52], dbits;
                        lds_q6(sdata + q6off + (uint32_t)((r * nb + j) * 210), L, dbits);
                        block_q6<NTOK>(L, dbits, xa, part);
                    }
                } else {
                    const XGlobal xa{M.x + (int64_t)b * 256, cols};
                    if (fmt == kFmtQ4K) {
                        uint4 v[9];
                        const uint32_t a = sdata + (uint32_t)(r * M.kb * 144 + j * 144);
#pragma unroll
                        for (int i = 0; i < 9; ++i) v[i] = lds_v4(a + 16 * i);
                        block_q45<NTOK, false>(v, xa, part);
                    } else if (fmt == kFmtQ5K) {
                        uint4 v[11];
                        const uint32_t a = sdata + (uint32_t)(r * M.kb * 176 + j * 176);
#pragma unroll
                        for (int i = 0; i < 11; ++i) v[i] = lds_v4(a + 16 * i);
                        block_q45<NTOK, true>(v, xa, part);
                    } else {
                        uint32_t L[52], dbits;
                        lds_q6(sdata + q6off + (uint32_t)((r * nb + j) * 210), L, dbits);
                        block_q6<NTOK>(L, dbits, xa, part);
                    }
                }
#pragma unroll
                for (int tt = 0; tt < NTOK; ++tt)
                    part_f[((size_t)r * nb + b) * NTOK + tt] = part[tt];
            }
        }
        batch_base += nbat;
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (kMaxSlots + slot));

        if (k == nbox - 1) {
            consumer_sync();  // every partial of group g is in shared memory
            const bool bad = *(volatile int *)&abort_flag;
#pragma unroll 1
            for (int o = threadIdx.x; o < h * NTOK; o += kStreamConsumers * 32) {
                const int r = o / NTOK, tt = o - (o / NTOK) * NTOK;
                float acc = part_f[((size_t)r * nb) * NTOK + tt];
#pragma unroll 1
                for (int b = 1; b < nb; ++b) acc += part_f[((size_t)r * nb + b) * NTOK + tt];
                M.y[(int64_t)tt * M.rows + g0 + r] = bad ? __int_as_float(0x7FC00000) : acc;
            }
            consumer_sync();  // partials may be overwritten by the next group
        }
    }
}

}  // namespace kq
