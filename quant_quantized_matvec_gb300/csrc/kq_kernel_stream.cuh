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

constexpr int kStreamConsumers = 12;
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
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 100000;\n"
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


// Word sources for Q6_K blocks staged in shared memory (kq_blocks.cuh).
struct Q6SharedAligned {
    const uint8_t *a;
    __device__ __forceinline__ void words4(int j, uint32_t (&o)[4]) const {
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = *reinterpret_cast<const uint32_t *>(a + 4 * (j + i));
    }
    __device__ __forceinline__ uint32_t dbits() const {
        return *reinterpret_cast<const uint16_t *>(a + 208);
    }
};
struct Q6SharedShifted {  // a = block start - 2 (4-byte aligned)
    const uint8_t *a;
    __device__ __forceinline__ void words4(int j, uint32_t (&o)[4]) const {
        uint32_t r[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) r[i] = *reinterpret_cast<const uint32_t *>(a + 4 * (j + i));
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(r[i], r[i + 1], 16);
    }
    __device__ __forceinline__ uint32_t dbits() const {
        return *reinterpret_cast<const uint32_t *>(a + 208) >> 16;
    }
};

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
    __shared__ int gcount[2];  // warps done with the row group of each buffer

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
    const uint32_t xbar = bars + 8 * (2 * kMaxSlots);  // inputs staged in shared memory
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < nslot; ++s) {
            mbar_init(bars + 8 * s, 1);
            mbar_init(bars + 8 * (kMaxSlots + s), kStreamConsumers);
        }
        mbar_init(xbar, 1);
        mbar_init(xbar + 8, 1);   // group reduction done, buffer 0
        mbar_init(xbar + 16, 1);  // group reduction done, buffer 1
        mbar_init(xbar + 24, kStreamConsumers);  // raw inputs consumed
        gcount[0] = gcount[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kStreamConsumers) {
        // ------------------------------------------------ producer
        if (lane != 0) return;
        // The raw inputs go first, into the last ring slot, which is not
        // filled with weights until the consumers have built their padded,
        // scaled copy of them.
        const uint32_t xraw = ring + (uint32_t)(nslot - 1) * p.slot_bytes;
        if (XSMEM) {
            const uint32_t xb = (uint32_t)(NTOK * (int64_t)nb * 256 * 4);
            mbar_expect_tx(xbar, xb);
            for (uint32_t o = 0; o < xb; o += 32768)
                bulk_g2s(xraw + o, reinterpret_cast<const uint8_t *>(M.x) + o,
                         xb - o < 32768 ? xb - o : 32768, xbar);
        }
        int issued = 0;
        int slot = 0, lap = 0, g = 0, k = 0;
        int64_t g0 = G.start(0), g1 = G.start(1);
        for (int s = 0; s < nstage; ++s) {
            if (XSMEM && s == nslot - 1) {
                if (*(volatile int *)&abort_flag) break;
                if (!mbar_wait(xbar + 24, 0)) {
                    atomicExch(&abort_flag, 1);
                    atomicOr(p.err, 1u);
                    break;
                }
            }
            if (s >= nslot) {
                if (*(volatile int *)&abort_flag) break;
                if (!mbar_wait(bars + 8 * (kMaxSlots + slot), (lap - 1) & 1)) {
                    atomicExch(&abort_flag, 1);
                    atomicOr(p.err, 1u);
                    break;
                }
            }
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
            if (++slot == nslot) {
                slot = 0;
                ++lap;
            }
            if (++k == nbox) {
                k = 0;
                ++g;
                g0 = g1;
                g1 = G.start(g + 1);
            }
        }
        if (*(volatile int *)&abort_flag) {
            // do not leave copies in flight into this CTA's shared memory
            if (XSMEM) mbar_wait(xbar, 0);
            for (int slot = 0; slot < nslot && slot < issued; ++slot) {
                const int last = slot + ((issued - 1 - slot) / nslot) * nslot;
                mbar_wait(bars + 8 * slot, (last / nslot) & 1);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int64_t cols = (int64_t)nb * 256;
    const bool q4 = fmt == kFmtQ4K;
    // scaled inputs, padded to 260 floats a block so that the inputs of
    // neighbouring block columns fall on different shared-memory banks
    const int xstride = nb * 260;
    const float *xs_f = reinterpret_cast<const float *>(smem + 1024);
    const float *xt_f = xs_f + NTOK * xstride;  // sub-block sums
    if (XSMEM) {
        // The producer copies x into the last ring slot first.  Take the
        // sub-block sums X_s from it (element order, as sum32 does from
        // global memory), and write the copy scaled for the bit position of
        // each weight's code (kq_blocks.cuh) into the padded layout.
        if (!mbar_wait(xbar, 0)) {
            atomicExch(&abort_flag, 1);
            atomicOr(p.err, 1u);
        }
        const float *xr = reinterpret_cast<const float *>(
            smem + (ring + (uint32_t)(nslot - 1) * p.slot_bytes - bars));
        float *xw = reinterpret_cast<float *>(smem + 1024);
        if (!q6) {
            float *tab = xw + NTOK * xstride;
            const int ns = (int)(NTOK * cols / 32);
            for (int i = threadIdx.x; i < ns; i += kStreamConsumers * 32) {
                const float4 *v4 = reinterpret_cast<const float4 *>(xr + 32 * i);
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 v = v4[j];
                    acc += v.x;
                    acc += v.y;
                    acc += v.z;
                    acc += v.w;
                }
                tab[i] = acc;
            }
        }
        const int n4 = (int)(NTOK * cols / 4);
        for (int i = threadIdx.x; i < n4; i += kStreamConsumers * 32) {
            const int e = (4 * i) & 255;  // cols is a multiple of 256
            const int blk = (4 * i) >> 8;  // token-major block index
            float4 v = reinterpret_cast<const float4 *>(xr)[i];
            v.x *= pow2f(xscale_exp(q4, e));
            v.y *= pow2f(xscale_exp(q4, e + 1));
            v.z *= pow2f(xscale_exp(q4, e + 2));
            v.w *= pow2f(xscale_exp(q4, e + 3));
            *reinterpret_cast<float4 *>(xw + blk * 260 + e) = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(xbar + 24);  // the raw copy may be overwritten
    }
    consumer_sync();

    // Row groups alternate between two partial buffers.  Each consumer warp
    // counts itself done with a group after the group's last stage; the last
    // warp to do so sums the group's partials in block order and writes y,
    // then releases the buffer (mbarrier) for the group two later.  No
    // consumer waits for the others at a group boundary.
    const int part_floats = p.part_bytes / 8;  // per buffer
    // A Q4_K / Q5_K task is one block column of two rows of the stage, p
    // and p + hp, which share their inputs; a Q6_K task is one row.
    const int rr = q6 ? 1 : 2;
    int batch_base = 0;
    int slot = 0, lap = 0, g = 0, k = 0;
    int64_t g0 = G.start(0), g1 = G.start(1);
    int h = (int)(g1 - g0);
    int hp = (h + rr - 1) / rr;
    uint32_t hinv = ((1u << 20) + (uint32_t)hp - 1) / (uint32_t)hp;
#pragma unroll 1
    for (int s = 0; s < nstage; ++s) {
        const int b0 = q6 ? 0 : k * M.kb;
        const int kbv = q6 ? nb : (nb - b0 < M.kb ? nb - b0 : M.kb);
        const int tasks = hp * kbv;
        const int nbat = (tasks + 31) / 32;
        const uint32_t sdata = ring + (uint32_t)slot * p.slot_bytes;
        const uint8_t *sdp = smem + (sdata - bars);
        float *pbuf = part_f + (g & 1) * part_floats;
        bool ok = !*(volatile int *)&abort_flag;
        if (ok && k == 0 && g >= 2 &&
            !mbar_wait(xbar + 8 + 8 * (g & 1), ((g >> 1) - 1) & 1)) {
            atomicExch(&abort_flag, 1);
            atomicOr(p.err, 1u);
            ok = false;
        }
        if (ok && !mbar_wait(bars + 8 * slot, lap & 1)) {
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
                // t / hp by multiply-shift: exact for t < 2^11, hp <= 32
                const int j = (int)(((uint32_t)t * hinv) >> 20), r = t - j * hp;
                const int b = b0 + j;
                const float *xsb = xs_f + b * 260;
                const float *xtb = xt_f + b * 8;
                const int xpl = xstride, spl = (int)(cols / 32);
                if (!q6) {
                    const int r2 = r + hp < h ? r + hp : h - 1;  // h odd: recompute, not stored
                    const int bb45 = fmt == kFmtQ4K ? 144 : 176;
                    const BlockShared B[2] = {
                        {reinterpret_cast<const uint4 *>(sdp + r * M.kb * bb45 + j * bb45)},
                        {reinterpret_cast<const uint4 *>(sdp + r2 * M.kb * bb45 + j * bb45)}};
                    float part[2][NTOK];
                    if (fmt == kFmtQ4K) {
                        if (XSMEM)
                            block_q45<NTOK, false, 2>(B, XSharedS{xsb, xpl, xtb, spl}, part);
                        else
                            block_q45<NTOK, false, 2>(B, XGlobalS<true>{M.x + (int64_t)b * 256, cols}, part);
                    } else {
                        if (XSMEM)
                            block_q45<NTOK, true, 2>(B, XSharedS{xsb, xpl, xtb, spl}, part);
                        else
                            block_q45<NTOK, true, 2>(B, XGlobalS<false>{M.x + (int64_t)b * 256, cols}, part);
                    }
#pragma unroll
                    for (int tt = 0; tt < NTOK; ++tt) {
                        pbuf[((size_t)r * nb + b) * NTOK + tt] = part[0][tt];
                        if (r + hp < h) pbuf[((size_t)r2 * nb + b) * NTOK + tt] = part[1][tt];
                    }
                } else {
                    float part[NTOK];
                    const uint8_t *a = sdp + q6off + (r * nb + j) * 210;
                    const bool shifted = (smem_addr(a) & 3u) != 0;
                    if (XSMEM) {
                        const XSharedS xa{xsb, xpl, xtb, spl};
                        if (shifted)
                            block_q6k<NTOK>(Q6SharedShifted{a - 2}, xa, part);
                        else
                            block_q6k<NTOK>(Q6SharedAligned{a}, xa, part);
                    } else {
                        const XGlobalS<false> xa{M.x + (int64_t)b * 256, cols};
                        if (shifted)
                            block_q6k<NTOK>(Q6SharedShifted{a - 2}, xa, part);
                        else
                            block_q6k<NTOK>(Q6SharedAligned{a}, xa, part);
                    }
#pragma unroll
                    for (int tt = 0; tt < NTOK; ++tt) pbuf[((size_t)r * nb + b) * NTOK + tt] = part[tt];
                }
            }
        }
        batch_base += nbat;
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (kMaxSlots + slot));

        if (k == nbox - 1) {
            // this warp is done with group g
            int old = 0;
            if (lane == 0) {
                __threadfence_block();
                old = atomicAdd(&gcount[g & 1], 1);
            }
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == kStreamConsumers - 1) {
                __threadfence_block();
                const bool bad = *(volatile int *)&abort_flag;
                if (lane < h) {
#pragma unroll 1
                    for (int tt = 0; tt < NTOK; ++tt) {
                        float acc = pbuf[((size_t)lane * nb) * NTOK + tt];
#pragma unroll 4
                        for (int b = 1; b < nb; ++b) acc += pbuf[((size_t)lane * nb + b) * NTOK + tt];
                        M.y[(int64_t)tt * M.rows + g0 + lane] = bad ? __int_as_float(0x7FC00000) : acc;
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    gcount[g & 1] = 0;
                    __threadfence_block();
                    mbar_arrive(xbar + 8 + 8 * (g & 1));
                }
            }
        }
        if (++slot == nslot) {
            slot = 0;
            ++lap;
        }
        if (++k == nbox) {
            k = 0;
            ++g;
            g0 = g1;
            g1 = G.start(g + 1);
            h = (int)(g1 - g0);
            hp = (h + rr - 1) / rr;
            hinv = hp > 0 ? ((1u << 20) + (uint32_t)hp - 1) / (uint32_t)hp : 1u;
        }
    }
}

}  // namespace kq
