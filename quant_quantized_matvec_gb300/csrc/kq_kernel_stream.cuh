// kq_kernel_stream.cuh -- the set kernel, TMA-streaming variant.
//
// One CTA per SM.  Each CTA owns a balanced, contiguous row range of one
// member of the set, split into row groups of at most 32 rows.  A producer
// warp streams the
// weights through a ring of shared-memory slots:
//   * Q4_K / Q5_K: one 2-D tensor-map box per stage, [h rows][kb blocks]
//     (kb chosen so that a box row is an odd number of 16-byte units and
//     rows land on distinct shared-memory banks), cp.async.bulk.tensor;
//   * Q6_K: rows are only 2-byte aligned (no tensor map), so the same
//     [h rows][kb blocks] stage is one 16-byte-aligned bulk copy
//     (cp.async.bulk) per row segment, segments M.seg bytes apart, the
//     sub-16-byte tail at the end of the matrix copied by the producer with
//     plain loads.
// The consumer warps, 12 (15 in the launch for tall Q6_K sets, NCW), turn
// the inputs into the fixed-point records of kq_xrec.cuh in shared memory
// (or read them from global memory, where a separate pass wrote them, when
// they do not fit).  Every consumer warp
// takes part in every stage: the stage's tasks -- one block column of two
// rows, p and p + hp, that share their inputs (of one row, RPT = 1, in the
// launch for tall Q6_K sets staged in row segments) -- ordered block-major
// so neighbouring lanes share inputs, are dealt out 32 at a time
// round-robin over the consumer warps; each lane turns its super-blocks
// into per-token partial sums (kq_blocks.cuh) stored in shared memory.  A
// row's partial is the same whichever rows share its task.  When a
// row group's last stage is done, the last warp to finish it sums each
// row's blocks in block order 0..nb-1 and writes y; the CTA's last group is
// summed the same way by all consumer warps together.  That sum order, and
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
#include "kq_tc.cuh"

namespace kq {

constexpr int kStreamConsumers = 12;
// Consumer warps of the one-token-column launch for Q6_K-only sets whose
// CTAs stream many stages (kq_api.cu, run_stream): 16 warps, 128
// registers each.  The Q6_K LM head 202048x6656 took 207.1 us per call
// with them against 216.1, FFN down Q6_K 6656x19968 36.3 against 37.3;
// other launches with 15 were slower (the QKV set 9.10 vs 8.85 us, the
// Q5_K LM head 164.9 vs 156.5).
constexpr int kStreamConsumersTall = 15;
constexpr int kMaxMaps = 4;
constexpr int kMaxSlots = 32;
constexpr int kOverlapPrefetch = 1;  // stages issued before the inputs (overlap)
constexpr int kMaxHinv = 40;  // row-pair offsets hp of a stage are at most 17
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s (default)

struct StreamMember {
    const uint8_t *W;
    const float *x;
    const uint8_t *rec;  // input records in global memory (when not staged);
                         // tensor-core launches: the records of kq_xtc.cuh
    float *y;
    int64_t rows;
    int32_t nb;
    int32_t fmt;
    int32_t cta_begin;
    int32_t ncta;
    int32_t rows_q, rows_r;  // rows / ncta, rows % ncta
    // row groups of a CTA with rows_q rows ([0]) or rows_q + 1 rows ([1]):
    // ng groups of gq or gq + 1 rows (the first gr one more)
    int32_t ng[2], gq[2], gr[2];
    int32_t rmax;   // rows per group at most
    int32_t kb;     // blocks per stage row
    int32_t seg;    // Q6_K: bytes between row segments in a slot
    int32_t q6_whole;  // Q6_K: stages of whole rows, one bulk copy each
    int32_t nmaps;  // tensor maps (box heights) for this member (Q4_K / Q5_K)
    int32_t map_h[kMaxMaps];
};

struct StreamParams {
    CUtensorMap maps[kMaxSet][kMaxMaps];
    StreamMember m[kMaxSet];
    int32_t n;
    int32_t nslot;
    int32_t slot_bytes;
    int32_t x_bytes;     // input records in shared memory (0: in global memory)
    int32_t part_bytes;
    int32_t part_bufs;   // partial buffers: 2, or 1 when no CTA has a second row group
    int32_t scr_bytes;   // tensor-core launches: per-warp unit scratch
    int32_t ntok;        // token columns of the launch (tensor-core launches
                         // are compiled for a multiple of 8)
    int32_t overlap;     // launched to overlap the preceding kernel
    uint32_t hinv[kMaxHinv + 1];  // ceil(2^20 / hp): t / hp = (t * hinv[hp]) >> 20
    unsigned int *err;   // device error word (nonzero: a wait expired)
    unsigned long long wait_ns;  // wall-time limit of each wait
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
// Wait for the phase of `parity` to complete; false once `limit_ns` of wall
// time have passed.  Between polls the thread sleeps, doubling from 32 ns up
// to `max_ns`, so that waiting warps leave the issue slots to working ones.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns,
                                          unsigned max_ns = 256) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    unsigned ns = 32;
    while (!mbar_try(bar, parity)) {
        __nanosleep(ns);
        if (ns < max_ns) ns <<= 1;
        if (global_ns() - t0 > limit_ns) return false;
    }
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
// Programmatic dependent launch: let the next kernel on the stream launch,
// and wait for the preceding one (no-ops for an ordinary launch).
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
template <int NCW>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
}

// Words of a Q6_K block staged in shared memory, 2-byte aligned: five
// aligned words funnel-shifted by 0 or 16 bits, the same instructions for
// either alignment (a warp's lanes do not split over the two).  The word
// after the block may be read (it lies inside the slot) and is discarded.
struct Q6WordsShared {
    const uint8_t *a4;  // block start rounded down to 4 bytes
    uint32_t sh;        // 8 * (block start - a4)
    static __device__ __forceinline__ Q6WordsShared at(const uint8_t *p) {
        // pointer arithmetic (not an integer round trip) keeps the
        // shared-memory address space visible, so the loads stay LDS
        const uint32_t mis = (uint32_t)reinterpret_cast<uintptr_t>(p) & 3u;
        return {p - mis, mis * 8u};
    }
    __device__ __forceinline__ void words4(int j, uint32_t (&o)[4]) const {
        uint32_t r[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) r[i] = reinterpret_cast<const uint32_t *>(a4)[j + i];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(r[i], r[i + 1], sh);
    }
    __device__ __forceinline__ uint32_t dbits() const {
        return *reinterpret_cast<const unsigned short *>(a4 + sh / 8 + 208);
    }
};

// Row-group geometry of a CTA: rows [ra, ra + n) split into ng groups of
// gq or gq + 1 rows (the first gr groups one more), without divisions in
// the stage loop.
struct Groups {
    int64_t ra;
    int n, ng, gq, gr;
    __device__ __forceinline__ int64_t start(int g) const {
        return ra + (int64_t)(g * gq + (g < gr ? g : gr));
    }
    // CTA cidx of member M, whose rows split into ncta CTAs of rows_q or
    // rows_q + 1 rows (the first rows_r CTAs one more); group splits are
    // precomputed on the host for both sizes
    template <class MEM>
    __device__ __forceinline__ void init(int cidx, const MEM &M) {
        const int big = cidx < M.rows_r ? 1 : 0;
        ra = (int64_t)cidx * M.rows_q + (big ? cidx : M.rows_r);
        n = M.rows_q + big;
        ng = M.ng[big];
        gq = M.gq[big];
        gr = M.gr[big];
    }
};

// Offset in a Q6_K stage slot of row r's block column b0 (`base` = the
// stage's first row's byte offset in W plus 210 b0; rows `rb` bytes long).
// Whole-row stages are one copy from the 16-byte boundary at or below the
// first row, so row r sits at (base mod 16) + r rb; row segments are
// `seg` bytes apart, each starting as far past a 16-byte boundary as its
// first block does in memory (the low four bits survive wrap-around).
__device__ __forceinline__ uint32_t q6_row_off(uint32_t base, int r, uint32_t rb, int seg,
                                               bool whole) {
    return whole ? (base & 15u) + (uint32_t)r * rb
                 : (uint32_t)(r * seg) + ((base + (uint32_t)r * rb) & 15u);
}

// Floats between rows of a partial buffer ([row][block][token]): one more
// than a row's nb x nt, an odd count, so that reads of one token from
// consecutive rows (the reductions) fall on distinct banks.
__host__ __device__ __forceinline__ int part_row_floats(int nb, int nt) { return nb * nt + 1; }

// Row pairs of a stage of h rows: rows p and p + hp for p < hp.
__device__ __forceinline__ int pair_offset(int h) { return (h + 1) >> 1; }

// Rows of one task: a lane takes one block column of R rows of the stage,
// p and p + hp, which share their inputs.  R = 2, except in the launch for
// tall Q6_K sets staged in row segments (kq_plan.h, stream_rows_per_lane),
// which takes R = 1: the template parameter RPT of kq_set_stream.
__host__ __device__ constexpr int stream_rows_per_task(int fmt, int ntok) {
    return (void)fmt, (void)ntok, 2;
}

// What the consumer warps share.
struct ConsumerCtx {
    uint8_t *smem;
    const float *x;       // inputs (records are built from them in shared memory)
    uint8_t *recs_w;      // shared-memory records to build
    int *xissued;         // consumer warps whose input loads have gone out
    const uint8_t *recs;  // this member's input records (shared or global)
    float *part_f;
    int part_step;        // floats from partial buffer 0 to 1 (0: one buffer)
    float *scr;           // tensor-core unit scratch (consumer warp 0's; then per warp)
    int scr_tiles;        // tiles of scales a warp's scratch holds (1 or 2)
    int ntok;
    uint32_t bars, ring, xbar;
    int nslot, slot_bytes;
    int nb, kb, nbox, nstage;
    int64_t rows, row_bytes;
    int q6_seg;
    bool q6_whole;
    float *y;
    Groups G;
    int *abort_flag;
    int *gcount;
    const uint32_t *hinv;  // ceil(2^20 / hp) by hp
    unsigned int *err;
    unsigned long long wait_ns;
};

// The CTA's last row group is summed by all consumer warps together once
// each is done with it (earlier groups are summed by the last warp to
// finish them, while the others go on): output (token tt, row r) is its nb
// block partials added in block order, as for every group.  `nt` = token
// columns of the partial buffer, `ntok` = token columns to store.
template <int NCW>
__device__ __forceinline__ void reduce_last_group(const ConsumerCtx &c, int nt, int ntok,
                                                  int warp, int lane) {
    consumer_sync<NCW>();
    const int gl = c.G.ng - 1;
    const int64_t g0 = c.G.start(gl);
    const int h = (int)(c.G.start(gl + 1) - g0);
    const float *pbuf = c.part_f + (gl & 1) * c.part_step;
    const bool bad = *(volatile int *)c.abort_flag;
    const int nb = c.nb;
#pragma unroll 1
    for (int o = warp * 32 + lane; o < h * ntok; o += NCW * 32) {
        const int tt = o / h, r = o - tt * h;
        const float *pp = pbuf + (int64_t)r * part_row_floats(nb, nt) + tt;
        float acc = pp[0];
#pragma unroll 4
        for (int bb = 1; bb < nb; ++bb) acc += pp[bb * nt];
        c.y[(int64_t)tt * c.rows + g0 + r] = bad ? __int_as_float(0x7FC00000) : acc;
    }
}

template <int NTOK, bool XSMEM, int FMT, int NCW, int RPT>
__device__ __forceinline__ void consume(const ConsumerCtx &c, int warp, int lane) {
    constexpr bool Q6 = FMT == kFmtQ6K;
    constexpr bool Q5 = FMT == kFmtQ5K;
    constexpr int BB = Q6 ? 210 : (Q5 ? 176 : 144);
    constexpr int REC = rec_bytes(Q6);
    constexpr int R = RPT;
    static_assert(R == 1 || R == 2, "one or two rows a task");
    using XR = Rec<!XSMEM>;
    const int nb = c.nb;
    const int tstride = nb * REC;
    const int prow = part_row_floats(nb, NTOK);
    if (XSMEM) {
        build_records<Q6>(c.x, (int64_t)nb * 256, NTOK, nb, c.recs_w, warp, NCW,
                          lane, [&] {
                              if (lane == 0)
                                  asm volatile("red.relaxed.cta.shared::cta.add.u32 [%0], 1;" ::"r"(
                                      smem_addr(c.xissued)));
                          });
        consumer_sync<NCW>();
    }
    int batch_base = 0;
    int rot = 0;  // batch_base % NCW
    int slot = 0, lap = 0, g = 0, k = 0;
    int64_t g0 = c.G.start(0), g1 = c.G.start(1);
    int h = (int)(g1 - g0);
    int hp = R == 2 ? pair_offset(h) : h;
    uint32_t hinv = c.hinv[hp];
#pragma unroll 1
    for (int s = 0; s < c.nstage; ++s) {
        const int b0 = k * c.kb;
        const int kbv = nb - b0 < c.kb ? nb - b0 : c.kb;
        const int tasks = hp * kbv;
        const int nbat = (int)(((uint32_t)tasks + 31u) >> 5);
        const uint8_t *sdp = c.smem + (c.ring - c.bars) + slot * c.slot_bytes;
        float *pbuf = c.part_f + (g & 1) * c.part_step;
        bool ok = !*(volatile int *)c.abort_flag;
        if (ok && k == 0 && g >= 2 &&
            !mbar_wait(c.xbar + 8 * (g & 1), ((g >> 1) - 1) & 1, c.wait_ns)) {
            atomicExch(c.abort_flag, 1);
            atomicOr(c.err, 1u);
            ok = false;
        }
        // Every warp waits for the slot, even one dealt no batch of this
        // stage: the wait keeps its arrival on the slot's empty barrier in
        // the right lap (a warp that skipped it could arrive for the slot's
        // next lap before this lap's readers are done, and the producer
        // would overwrite the slot under them).
        if (ok && !mbar_wait(c.bars + 8 * slot, lap & 1, c.wait_ns, 128)) {
            atomicExch(c.abort_flag, 1);
            atomicOr(c.err, 1u);
            ok = false;
        }
        if (ok) {
            // this warp's first batch: the one dealt to it in the rotation
            int dw = warp - rot;
            if (dw < 0) dw += NCW;
            int bat = batch_base + dw;
#pragma unroll 1
            for (; bat < batch_base + nbat; bat += NCW) {
                // Lanes past the stage's last task redo the last task and do
                // not store it: the whole warp runs the block code together,
                // which keeps its loops warp-uniform.
                const int tl = (bat - batch_base) * 32 + lane;
                const bool valid = tl < tasks;
                const int t = valid ? tl : tasks - 1;
                // t / hp by multiply-shift: exact for t < 2^12, hp <= 32 (the
                // planner keeps every stage below 2^12 tasks)
                const int j = (int)(((uint32_t)t * hinv) >> 20), r = t - j * hp;
                const int r2 = (R == 2 && r + hp < h) ? r + hp : r;
                const int b = b0 + j;
                const XR xr{c.recs + b * REC, tstride};
                float part[R][NTOK];
                if (!Q6) {
                    BlockShared B[R];
                    B[0].p = reinterpret_cast<const uint4 *>(sdp + (r * c.kb + j) * BB);
                    if (R == 2) B[R - 1].p = reinterpret_cast<const uint4 *>(sdp + (r2 * c.kb + j) * BB);
                    block_q45<NTOK, Q5, R>(B, xr, part);
                } else {
                    // one code path for every lane, whatever its blocks'
                    // alignment: row r's segment starts as far past a
                    // 16-byte boundary as its first block does in memory
                    // block start (row g0 + r, block b0) mod 16: the low four
                    // bits survive 32-bit wrap-around
                    const uint32_t base = (uint32_t)g0 * (uint32_t)c.row_bytes + (uint32_t)b0 * 210u;
                    const uint32_t rb = (uint32_t)c.row_bytes;
                    const uint8_t *a0 = sdp + q6_row_off(base, r, rb, c.q6_seg, c.q6_whole) + j * 210;
                    const uint8_t *a1 = sdp + q6_row_off(base, r2, rb, c.q6_seg, c.q6_whole) + j * 210;
                    Q6WordsShared W[R];
                    W[0] = Q6WordsShared::at(a0);
                    if (R == 2) W[R - 1] = Q6WordsShared::at(a1);
                    block_q6k<NTOK, R>(W, xr, part);
                }
                if (valid) {
#pragma unroll
                    for (int tt = 0; tt < NTOK; ++tt) {
                        pbuf[r * prow + b * NTOK + tt] = part[0][tt];
                        if (R == 2 && r2 != r) pbuf[r2 * prow + b * NTOK + tt] = part[R - 1][tt];
                    }
                }
            }
        }
        batch_base += nbat;
        rot += nbat;
        while (rot >= NCW) rot -= NCW;
        __syncwarp();
        if (lane == 0) mbar_arrive(c.bars + 8 * (kMaxSlots + slot));

        if (k == c.nbox - 1 && g < c.G.ng - 1) {
            // this warp is done with group g
            int old = 0;
            if (lane == 0) {
                __threadfence_block();
                old = atomicAdd(&c.gcount[g & 1], 1);
            }
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == NCW - 1) {
                __threadfence_block();
                const bool bad = *(volatile int *)c.abort_flag;
                if (lane < h) {
#pragma unroll 1
                    for (int tt = 0; tt < NTOK; ++tt) {
                        float acc = pbuf[lane * prow + tt];
#pragma unroll 4
                        for (int bb = 1; bb < nb; ++bb) acc += pbuf[lane * prow + bb * NTOK + tt];
                        c.y[(int64_t)tt * c.rows + g0 + lane] =
                            bad ? __int_as_float(0x7FC00000) : acc;
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    c.gcount[g & 1] = 0;
                    __threadfence_block();
                    mbar_arrive(c.xbar + 8 * (g & 1));
                }
            }
        }
        if (++slot == c.nslot) {
            slot = 0;
            ++lap;
        }
        if (++k == c.nbox) {
            k = 0;
            ++g;
            g0 = g1;
            g1 = c.G.start(g + 1);
            h = (int)(g1 - g0);
            hp = h < 1 ? 1 : (R == 2 ? pair_offset(h) : h);
            hinv = c.hinv[hp];
        }
    }
    reduce_last_group<NCW>(c, NTOK, NTOK, warp, lane);
}

// One unit of a tensor-core launch: block column j of the stage (column
// b0 + j of the rows) for rows r0.. of the group's h rows as MT 16-row
// tiles, its partials stored in pbuf.  `base`: the Q6_K stage's first row
// offset (see q6_row_off).
template <int FMT, int NOCT, int MT>
__device__ __forceinline__ void tc_column(const ConsumerCtx &c, const uint8_t *sdp, uint32_t base,
                                          int b0, int j, int r0, int h, const uint8_t *col,
                                          float *scr, float *pbuf, int lane) {
    constexpr bool Q6 = FMT == kFmtQ6K;
    constexpr int BB = Q6 ? 210 : (FMT == kFmtQ5K ? 176 : 144);
    constexpr int NT = 8 * NOCT;
    const int prow = part_row_floats(c.nb, NT);
    const int nvalid = h - r0 < 16 * MT ? h - r0 : 16 * MT;
    float v[MT][NOCT][2][2];
    if (!Q6) {
        const uint8_t *blk = sdp + r0 * (c.kb * BB) + j * BB;
        const int rs = c.kb * BB;
        tc_unit_mt<FMT, NOCT, false, true, MT>([&](int r) { return blk + r * rs; }, nvalid, col,
                                               c.ntok, scr, lane, v);
    } else {
        const uint32_t rb = (uint32_t)c.row_bytes;
        tc_unit_mt<FMT, NOCT, false, true, MT>(
            [&](int r) {
                return sdp + q6_row_off(base, r0 + r, rb, c.q6_seg, c.q6_whole) + j * 210;
            },
            nvalid, col, c.ntok, scr, lane, v);
    }
    const int gg = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
            const int row = r0 + 16 * m + gg + 8 * k2;
            if (row < h) {
#pragma unroll
                for (int o = 0; o < NOCT; ++o)
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj)
                        pbuf[row * prow + (b0 + j) * NT + 8 * o + 2 * t4 + jj] = v[m][o][k2][jj];
            }
        }
}

// The consumer of a tensor-core launch (ntok >= kTcMinNtok, any format):
// the stage's work is cut into units of one block column of one 16-row
// tile, or of both tiles of a 32-row group with two octets of tokens
// (tc_unit_tiles; kq_tc.cuh, all NOCT octets at once), and the CTA's whole
// sequence of units, stage after stage, is dealt round-robin: warp w takes
// units w, w + kStreamConsumers, ...  Each warp still waits for every
// stage's slot and arrives on its empty barrier once per stage (see
// consume).  The input records (kq_xtc.cuh) are read from global memory
// (L2, then L1).
template <int NOCT, int FMT>
__device__ __forceinline__ void consume_tc(const ConsumerCtx &c, int warp, int lane) {
    constexpr int NT = 8 * NOCT;
    const int nb = c.nb;
    const int prow = part_row_floats(nb, NT);
    constexpr int MT = tc_unit_tiles(NOCT);
    float *scr = c.scr + warp * c.scr_tiles * (kTcScrBytes / 4);
    constexpr int colb = tc_col_bytes(NOCT);
    int next = warp;  // this warp's next unit, counted over the whole CTA
    int ubase = 0;    // units of the stages before this one
    int slot = 0, lap = 0, g = 0, k = 0;
    int64_t g0 = c.G.start(0), g1 = c.G.start(1);
    int h = (int)(g1 - g0);
#pragma unroll 1
    for (int s = 0; s < c.nstage; ++s) {
        const int b0 = k * c.kb;
        const int kbv = nb - b0 < c.kb ? nb - b0 : c.kb;
        const int tiles = (h + 15) >> 4;  // 1 or 2
        // one unit spans both tiles (the scratch holds both tiles' scales)
        const bool pair = MT == 2 && tiles == 2 && c.scr_tiles == 2;
        const int units = (pair ? 1 : tiles) * kbv;
        const uint8_t *sdp = c.smem + (c.ring - c.bars) + slot * c.slot_bytes;
        float *pbuf = c.part_f + (g & 1) * c.part_step;
        bool ok = !*(volatile int *)c.abort_flag;
        if (ok && k == 0 && g >= 2 &&
            !mbar_wait(c.xbar + 8 * (g & 1), ((g >> 1) - 1) & 1, c.wait_ns)) {
            atomicExch(c.abort_flag, 1);
            atomicOr(c.err, 1u);
            ok = false;
        }
        if (ok && !mbar_wait(c.bars + 8 * slot, lap & 1, c.wait_ns, 128)) {
            atomicExch(c.abort_flag, 1);
            atomicOr(c.err, 1u);
            ok = false;
        }
        // Q6_K: a row segment starts as far past a 16-byte boundary as its
        // first block does in memory (low four bits survive wrap-around)
        const uint32_t base = (uint32_t)g0 * (uint32_t)c.row_bytes + (uint32_t)b0 * 210u;
#pragma unroll 1
        for (; next < ubase + units; next += kStreamConsumers) {
            if (!ok) continue;
            const int ul = next - ubase;
            // block column within the stage, first row of the unit
            const int j = (!pair && tiles == 2) ? ul >> 1 : ul;
            const int r0 = (!pair && tiles == 2) ? (ul & 1) * 16 : 0;
            const uint8_t *col = c.recs + (int64_t)(b0 + j) * colb;  // column b0 + j's records
            if (pair)
                tc_column<FMT, NOCT, MT>(c, sdp, base, b0, j, 0, h, col, scr, pbuf, lane);
            else
                tc_column<FMT, NOCT, 1>(c, sdp, base, b0, j, r0, h, col, scr, pbuf, lane);
        }
        ubase += units;
        __syncwarp();
        if (lane == 0) mbar_arrive(c.bars + 8 * (kMaxSlots + slot));

        if (k == c.nbox - 1 && g < c.G.ng - 1) {
            // this warp is done with group g
            int old = 0;
            if (lane == 0) {
                __threadfence_block();
                old = atomicAdd(&c.gcount[g & 1], 1);
            }
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == kStreamConsumers - 1) {
                __threadfence_block();
                const bool bad = *(volatile int *)c.abort_flag;
                if (lane < h) {
#pragma unroll 1
                    for (int tt = 0; tt < c.ntok; ++tt) {
                        float acc = pbuf[lane * prow + tt];
#pragma unroll 4
                        for (int bb = 1; bb < nb; ++bb) acc += pbuf[lane * prow + bb * NT + tt];
                        c.y[(int64_t)tt * c.rows + g0 + lane] =
                            bad ? __int_as_float(0x7FC00000) : acc;
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    c.gcount[g & 1] = 0;
                    __threadfence_block();
                    mbar_arrive(c.xbar + 8 * (g & 1));
                }
            }
        }
        if (++slot == c.nslot) {
            slot = 0;
            ++lap;
        }
        if (++k == c.nbox) {
            k = 0;
            ++g;
            g0 = g1;
            g1 = c.G.start(g + 1);
            h = (int)(g1 - g0);
        }
    }
    reduce_last_group<kStreamConsumers>(c, NT, c.ntok, warp, lane);
}

template <int NTOK, bool XSMEM, bool TC, int NCW = kStreamConsumers, int RPT = 2>
__global__ void __launch_bounds__(32 * (NCW + 1), 1)
    kq_set_stream(const __grid_constant__ StreamParams p) {
    static_assert(!TC || (NTOK % 8 == 0 && !XSMEM), "tensor-core launches: octets, global records");
    static_assert(!TC || NCW == kStreamConsumers, "tensor-core launches: the scratch is sized for 12 warps");
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int abort_flag;
    __shared__ int gcount[2];  // warps done with the row group of each buffer
    __shared__ int xissued;    // consumer warps whose input loads have gone out

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
    G.init(cidx, M);
    const bool q6 = fmt == kFmtQ6K;
    const int nbox = (nb + M.kb - 1) / M.kb;
    const int nstage = G.ng * nbox;
    const int nslot = p.nslot;

    const uint32_t bars = smem_addr(smem);  // full[0..kMaxSlots), empty[..]
    const uint32_t recs = bars + 1024;
    const uint32_t parts = recs + p.x_bytes;
    const uint32_t scrs = parts + p.part_bytes;
    const uint32_t ring = scrs + p.scr_bytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t xbar = bars + 8 * (2 * kMaxSlots);  // row group reduced, buffers 0 / 1
    allow_dependents();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < nslot; ++s) {
            mbar_init(bars + 8 * s, 1);
            mbar_init(bars + 8 * (kMaxSlots + s), NCW);
        }
        mbar_init(xbar, 1);
        mbar_init(xbar + 8, 1);
        gcount[0] = gcount[1] = 0;
        xissued = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------------------------ producer
        // Lane 0 takes every decision and every wait and shares the outcome
        // with the warp; the other lanes only help issue Q6_K row-segment
        // copies (lane r copies rows r, r + 32, ...).
        constexpr unsigned kAll = 0xFFFFFFFFu;
        // The consumers' input loads must not queue behind the weight
        // stream.  The producer issues `gate` stages, then waits until every
        // consumer warp is about to issue its input loads (a relaxed
        // counter) before it issues the rest.  gate = 0 for an ordinary
        // launch; with launch overlap a few stages go out first, while the
        // consumers still wait for the preceding kernel.
        const int gate = XSMEM ? (p.overlap ? kOverlapPrefetch : 0) : -1;
        auto wait_inputs_issued = [&]() {
            if (lane == 0) {
                const unsigned long long t0 = global_ns();
                while (*(volatile int *)&xissued < NCW) {
                    __nanosleep(20);
                    if (global_ns() - t0 > p.wait_ns) {
                        atomicExch(&abort_flag, 1);
                        atomicOr(p.err, 1u);
                        break;
                    }
                }
            }
            __syncwarp();
        };
        if (gate == 0) wait_inputs_issued();
        int issued = 0;
        int slot = 0, lap = 0, g = 0, k = 0;
        int64_t g0 = G.start(0), g1 = G.start(1);
        for (int s = 0; s < nstage; ++s) {
            if (s == gate && s > 0) wait_inputs_issued();
            int stop = 0;
            if (lane == 0) {
                stop = *(volatile int *)&abort_flag;
                if (!stop && s >= nslot &&
                    !mbar_wait(bars + 8 * (kMaxSlots + slot), (lap - 1) & 1, p.wait_ns)) {
                    atomicExch(&abort_flag, 1);
                    atomicOr(p.err, 1u);
                    stop = 1;
                }
                // Read the flag again after the slot became free: if every
                // consumer warp gave up on this slot's last stage, they set
                // the flag before arriving, and that stage's copy may still
                // be landing -- the slot must not be given a second copy.
                // (If any warp waited successfully, the copy has landed.)
                if (!stop) stop = *(volatile int *)&abort_flag;
            }
            if (__shfl_sync(kAll, stop, 0)) break;
            const int h = (int)(g1 - g0);
            const uint32_t dst = ring + (uint32_t)slot * p.slot_bytes;
            const uint32_t full = bars + 8 * slot;
            if (!q6) {
                if (lane == 0) {
                    int mj = 0;
                    for (int j = 0; j < M.nmaps; ++j)
                        if (M.map_h[j] == h) mj = j;
                    const int box_row = M.kb * bb;
                    mbar_expect_tx(full, (uint32_t)(h * box_row));
                    tensor2d_g2s(dst, &p.maps[mi][mj], k * (box_row / 8), (int)g0, full);
                }
            } else if (M.q6_whole) {
                // one 16-byte-aligned bulk copy of the stage's whole rows;
                // the sub-16-byte tail at the very end of the matrix is
                // copied with plain loads
                if (lane == 0) {
                    const int64_t total = M.rows * row_bytes;
                    const int64_t a = g0 * row_bytes, e = (g0 + h) * row_bytes;
                    const int64_t a16 = a & ~(int64_t)15;
                    int64_t e16 = (e + 15) & ~(int64_t)15;
                    if (e16 > total) {
                        e16 = total & ~(int64_t)15;
                        uint8_t *dstp = smem + (dst - bars);
                        for (int64_t i = e16; i < e; ++i) dstp[i - a16] = M.W[i];
                    }
                    // the tail's plain stores precede this arrive (a release)
                    mbar_expect_tx(full, (uint32_t)(e16 - a16));
                    bulk_g2s(dst, M.W + a16, (uint32_t)(e16 - a16), full);
                }
            } else {
                // one 16-byte-aligned bulk copy per row segment (blocks
                // b0..b0+kbv of the row), segments M.seg bytes apart; the
                // sub-16-byte tail at the very end of the matrix is copied
                // with plain loads
                const int64_t total = M.rows * row_bytes;
                const int b0 = k * M.kb;
                const int kbv = nb - b0 < M.kb ? nb - b0 : M.kb;
                uint8_t *dstp = smem + (dst - bars);
                uint32_t tx = 0;
                for (int r = lane; r < h; r += 32) {
                    const int64_t a = (g0 + r) * row_bytes + (int64_t)b0 * 210;
                    const int64_t e = a + (int64_t)kbv * 210;
                    const int64_t a16 = a & ~(int64_t)15;
                    int64_t e16 = (e + 15) & ~(int64_t)15;
                    if (e16 > total) {
                        e16 = total & ~(int64_t)15;
                        for (int64_t i = e16; i < e; ++i) dstp[r * M.seg + (i - a16)] = M.W[i];
                    }
                    tx += (uint32_t)(e16 - a16);
                }
                tx = __reduce_add_sync(kAll, tx);
                // the tail's plain stores are ordered before lane 0's
                // arrive (a release) by the warp barrier
                __syncwarp();
                if (lane == 0) mbar_expect_tx(full, tx);
                __syncwarp();
                for (int r = lane; r < h; r += 32) {
                    const int64_t a = (g0 + r) * row_bytes + (int64_t)b0 * 210;
                    const int64_t e = a + (int64_t)kbv * 210;
                    const int64_t a16 = a & ~(int64_t)15;
                    int64_t e16 = (e + 15) & ~(int64_t)15;
                    if (e16 > total) e16 = total & ~(int64_t)15;
                    bulk_g2s(dst + (uint32_t)(r * M.seg), M.W + a16, (uint32_t)(e16 - a16), full);
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
        __syncwarp();
        if (lane == 0 && *(volatile int *)&abort_flag) {
            // do not leave copies in flight into this CTA's shared memory
            // (always the default limit: copies that were issued do land)
            for (int slot = 0; slot < nslot && slot < issued; ++slot) {
                const int last = slot + ((issued - 1 - slot) / nslot) * nslot;
                mbar_wait(bars + 8 * slot, (last / nslot) & 1, kWaitLimitNs);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    // x (or its records) and y belong to the stream order: with an
    // overlapping launch, wait for the preceding kernel first.
    wait_prerequisites();
    ConsumerCtx c;
    c.x = M.x;
    c.xissued = &xissued;
    c.smem = smem;
    c.recs = XSMEM ? smem + (recs - bars) : M.rec;
    c.recs_w = smem + (recs - bars);
    c.part_f = reinterpret_cast<float *>(smem + (parts - bars));
    c.part_step = p.part_bufs == 2 ? p.part_bytes / 8 : 0;
    c.scr = reinterpret_cast<float *>(smem + (scrs - bars));
    c.scr_tiles = p.scr_bytes >= NCW * 2 * kTcScrBytes ? 2 : 1;
    c.ntok = p.ntok;
    c.bars = bars;
    c.ring = ring;
    c.xbar = xbar;
    c.nslot = nslot;
    c.slot_bytes = p.slot_bytes;
    c.nb = nb;
    c.kb = M.kb;
    c.nbox = nbox;
    c.nstage = nstage;
    c.rows = M.rows;
    c.row_bytes = row_bytes;
    c.q6_seg = M.seg;
    c.q6_whole = M.q6_whole != 0;
    c.y = M.y;
    c.G = G;
    c.abort_flag = &abort_flag;
    c.gcount = gcount;
    c.err = p.err;
    c.wait_ns = p.wait_ns;
    c.hinv = p.hinv;
    if constexpr (TC) {
        if (fmt == kFmtQ4K)
            consume_tc<NTOK / 8, kFmtQ4K>(c, warp, lane);
        else if (fmt == kFmtQ5K)
            consume_tc<NTOK / 8, kFmtQ5K>(c, warp, lane);
        else
            consume_tc<NTOK / 8, kFmtQ6K>(c, warp, lane);
    } else {
        if (fmt == kFmtQ4K)
            consume<NTOK, XSMEM, kFmtQ4K, NCW, RPT>(c, warp, lane);
        else if (fmt == kFmtQ5K)
            consume<NTOK, XSMEM, kFmtQ5K, NCW, RPT>(c, warp, lane);
        else
            consume<NTOK, XSMEM, kFmtQ6K, NCW, RPT>(c, warp, lane);
    }
}

}  // namespace kq
