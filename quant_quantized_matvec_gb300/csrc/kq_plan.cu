// kq_plan.cu -- launch geometry of the streaming kernel (host only).
#include "kq_plan.h"

#include <stdint.h>

#include <algorithm>

#include "kq_internal.h"
#include "kq_kernel_stream.cuh"
#include "kq_xrec.cuh"

namespace kqplan {

namespace {

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

int64_t block_bytes(int fmt) { return fmt == KQ_Q4_K ? 144 : fmt == KQ_Q5_K ? 176 : 210; }

// CTAs per member in proportion to its work (at least one, at most one per
// row), largest remainder first.  Work is bytes weighted by the format's
// consumer cost per byte relative to Q4_K.
void split_ctas(const kq_mat *mats, int n, int G, int *ncta) {
    int64_t bytes[KQ_MAX_SET], total = 0;
    for (int i = 0; i < n; ++i) {
        bytes[i] = mats[i].rows * (mats[i].cols / 256) * block_bytes(mats[i].fmt);
        if (mats[i].fmt == KQ_Q6_K) bytes[i] = bytes[i] * kCostQ6 / 16;
        total += bytes[i];
    }
    double rem[KQ_MAX_SET];
    int used = 0;
    for (int i = 0; i < n; ++i) {
        const double share = (double)G * (double)bytes[i] / (double)total;
        ncta[i] = std::max(1, (int)share);
        rem[i] = share - (int)share;
        ncta[i] = (int)std::min<int64_t>(ncta[i], mats[i].rows);
        used += ncta[i];
    }
    while (used < G) {
        int best = -1;
        for (int i = 0; i < n; ++i)
            if (ncta[i] < mats[i].rows && (best < 0 || rem[i] > rem[best])) best = i;
        if (best < 0) break;
        ++ncta[best];
        rem[best] = -1.0;
        ++used;
    }
    while (used > G) {  // only when n > G
        int best = 0;
        for (int i = 1; i < n; ++i)
            if (ncta[i] > ncta[best]) best = i;
        if (ncta[best] <= 1) break;
        --ncta[best];
        --used;
    }
}

// Q6_K: bytes between row segments in a slot.  A segment of kb blocks
// starts up to 14 bytes past a 16-byte boundary and its copy ends up to 14
// bytes past its end; an odd number of 16-byte units puts consecutive rows
// on different banks.
int q6_seg(int kb) {
    int seg = (int)round_up((int64_t)kb * 210 + 28, 16);
    if (((seg / 16) & 1) == 0) seg += 16;
    return seg;
}

// Weight bytes of a stage slot: h rows of kb blocks.
int64_t stage_weight_bytes(int fmt, int h, int kb) {
    return fmt == KQ_Q6_K ? (int64_t)h * q6_seg(kb) : (int64_t)h * kb * block_bytes(fmt);
}

// Q6_K rows of at most this many bytes are staged whole: a stage is a run
// of consecutive rows, one contiguous bulk copy (their bytes plus up to 15
// before and after for 16-byte alignment).  Longer rows are staged in
// per-row segments of kb blocks, so that a stage still holds enough rows.
constexpr int64_t kQ6WholeRowMax = 8192;

int64_t q6_whole_bytes(int h, int64_t row_bytes) { return round_up(h * row_bytes + 30, 16); }

// Stage geometry levels, from the largest stages down: stages are
// [h rows][kb blocks] with h <= rcap and stage rows of at most kb_bytes.
constexpr int kLevelRcap[] = {32, 16, 16, 8, 8};
constexpr int kLevelKbBytes[] = {2048, 2048, 1024, 1024, 512};
constexpr int kLevels = 5;

// The geometry of one level (x_bytes: records in shared memory).
kq_status plan_level(const kq_mat *mats, int n, int ntok, const int *ncta, int level, Plan &P) {
    const int rcap = kLevelRcap[level], kb_bytes = kLevelKbBytes[level];
    const bool tc = P.tc_noct > 0;
    const int ntok_part = tc ? 8 * P.tc_noct : ntok;  // token columns of the partials
    P.x_bytes = P.part_bytes = P.slot_bytes = P.stages = P.scr_bytes = 0;
    P.part_bufs = 1;
    int cta = 0;
    for (int i = 0; i < n; ++i) {
        const kq_mat &m = mats[i];
        Member &M = P.m[i];
        M = Member{};
        const int nb = (int)(m.cols / 256);
        const int bb = (int)block_bytes(m.fmt);
        M.row_bytes = (int64_t)nb * bb;
        M.cta_begin = cta;
        M.ncta = ncta[i];
        M.rows_q = (int)(m.rows / ncta[i]);
        M.rows_r = (int)(m.rows % ncta[i]);
        cta += ncta[i];
        // rows per group: partials for the group must fit in 64 KiB
        const int64_t part_row = (int64_t)kq::part_row_floats(nb, ntok_part) * 4;
        int rmax = (int)std::min<int64_t>(64 * 1024 / part_row, rcap);
        if (rmax < 1) return KQ_ERR_SHAPE;
        // Whole Q6_K rows (dp4a launches): a stage is one group of about
        // kb_bytes x rcap bytes of consecutive rows.  Taken when a CTA's
        // rows fit in one such stage, or make many groups of row segments
        // anyway (eight or more: the LM head's 1329 rows per CTA); in
        // between, whole-row stages split a few segment groups into more
        // (measured slower at 27 rows per CTA on Q6_K 4096x6656: 9.20 vs
        // 8.44 us at ntok 1, 19.05 vs 15.87 us at ntok 3).  Tensor-core
        // launches keep segments: their units read every stage's columns'
        // input fragments, which whole-row stages of few rows would
        // multiply.
        if (!tc && m.fmt == KQ_Q6_K && M.row_bytes <= kQ6WholeRowMax) {
            const int hw = (int)std::max<int64_t>(
                1, std::min<int64_t>(rmax, (int64_t)kb_bytes * rcap / M.row_bytes));
            const int64_t cta_rows = M.rows_q + (M.rows_r > 0 ? 1 : 0);
            // ... and only in stages of 8 or more rows: the LM head at 3
            // token columns (16-row groups, 6-row whole-row stages) took
            // 547 us against 406 with row segments
            if (hw >= 8 && (cta_rows <= hw || cta_rows >= 8 * (int64_t)rmax)) {
                M.whole = 1;
                rmax = hw;
            }
        }
        M.rmax = rmax;
        for (int big = 0; big < 2; ++big) {  // CTAs of rows_q / rows_q + 1 rows
            const int64_t nn = M.rows_q + big;
            const int64_t ng = nn > 0 ? (nn + rmax - 1) / rmax : 1;
            M.ng[big] = (int)ng;
            M.gq[big] = (int)(nn / ng);
            M.gr[big] = (int)(nn % ng);
        }
        // group heights that occur: n in {floor, ceil}(rows / ncta)
        const int64_t nlo = m.rows / ncta[i], nhi = (m.rows + ncta[i] - 1) / ncta[i];
        for (int64_t nn = nlo; nn <= nhi; ++nn) {
            if (nn < 1) continue;
            const int64_t ng = (nn + rmax - 1) / rmax;
            for (int64_t hh = nn / ng; hh <= (nn + ng - 1) / ng; ++hh) {
                bool seen = false;
                for (int j = 0; j < M.nh; ++j) seen |= M.hs[j] == hh;
                if (!seen) {
                    if (M.nh == kMaxHeights) return KQ_ERR_SHAPE;
                    M.hs[M.nh++] = (int)hh;
                }
                M.hmax = std::max<int>(M.hmax, (int)hh);
            }
        }
        // Blocks per stage row: at most kb_bytes (and 256 u64); prefer few
        // stages per row, then no zero-filled tail, then an odd number of
        // 16-byte units per row (rows on distinct banks).
        {
            const int kbmax = (int)std::max<int64_t>(1, std::min<int64_t>(nb, kb_bytes / bb));
            int best = 0;
            int64_t best_key = INT64_MAX;
            for (int kb = 1; kb <= kbmax; ++kb) {
                const int64_t nbox = (nb + kb - 1) / kb, waste = nbox * kb - nb;
                const int64_t units = (int64_t)kb * bb / 16;
                const int64_t key = nbox * 1000000 + waste * 10 + ((units & 1) ? 0 : 1);
                if (key < best_key) {
                    best_key = key;
                    best = kb;
                }
            }
            if (best == 0) return KQ_ERR_SHAPE;
            M.kb = M.whole ? nb : best;
        }
        // dp4a launches: tasks of a stage (row pairs x block columns) stay
        // below 2^12, the range of the kernel's multiply-shift division
        if (!tc) {
            const int hp = kq::stream_rows_per_task(m.fmt, ntok) == 2 ? (M.hmax + 1) / 2 : M.hmax;
            if ((int64_t)hp * M.kb >= 4096) return KQ_ERR_SHAPE;
        }
        if (m.fmt == KQ_Q6_K) M.seg = M.whole ? (int)M.row_bytes : q6_seg(M.kb);
        P.slot_bytes = std::max<int64_t>(
            P.slot_bytes, M.whole ? q6_whole_bytes(M.hmax, M.row_bytes)
                                  : stage_weight_bytes(m.fmt, M.hmax, M.kb));
        // CTAs of rows_q (+ 1) rows exist when rows_r < ncta (rows_r > 0)
        if ((M.rows_r < M.ncta && M.ng[0] > 1) || (M.rows_r > 0 && M.ng[1] > 1)) P.part_bufs = 2;
        // stages of this member's largest CTA
        P.stages = std::max<int64_t>(P.stages, (int64_t)M.ng[M.rows_r > 0 ? 1 : 0] *
                                                   ((nb + M.kb - 1) / M.kb));
        // input records [ntok][nb] (kq_xrec.cuh); tensor-core launches read
        // theirs from global memory
        if (!tc)
            P.x_bytes = std::max<int64_t>(P.x_bytes, (int64_t)ntok * nb * kq::rec_bytes(m.fmt == KQ_Q6_K));
        P.part_bytes = std::max<int64_t>(P.part_bytes, (int64_t)M.hmax * part_row);
    }
    // two row groups in flight (dp4a launches always; tensor-core launches
    // where a CTA has a second group)
    if (!tc) P.part_bufs = 2;
    P.part_bytes = P.part_bufs * round_up(P.part_bytes, 128);
    P.slot_bytes = round_up(P.slot_bytes, 128);
    P.x_bytes = round_up(P.x_bytes, 128);
    // tensor-core launches: each consumer warp's unit scratch, two tiles'
    // scales where units span two tiles (groups of more than 16 rows)
    if (tc) {
        int64_t hmax = 0;
        for (int i = 0; i < n; ++i) hmax = std::max<int64_t>(hmax, P.m[i].hmax);
        const int tiles = hmax > 16 ? kq::tc_unit_tiles(P.tc_noct) : 1;
        P.scr_bytes = round_up((int64_t)kq::kStreamConsumers * tiles * kq::kTcScrBytes, 128);
    }
    P.grid = cta;
    return KQ_OK;
}

}  // namespace

kq_status plan_stream(const kq_mat *mats, int n, int ntok, int sms, int smem_optin, Plan *out,
                      int tc_noct) {
    Plan &P = *out;
    P = Plan{};
    P.n = n;
    P.ntok = ntok;
    P.tc_noct = tc_noct;
    int ncta[KQ_MAX_SET];
    split_ctas(mats, n, sms, ncta);
    // The first level whose input records fit in shared memory beside at
    // least three slots (two at the smallest level, or when a CTA has only
    // two stages) is taken; if none fits, level 0 with the records in
    // global memory.  The 1 KiB alignment of the dynamic region pads the
    // static part to 1 KiB.
    const int64_t budget = (int64_t)smem_optin - 1024;
    for (int L = 0; L < kLevels && P.level < 0 && tc_noct == 0; ++L) {
        if (plan_level(mats, n, ntok, ncta, L, P) != KQ_OK) continue;
        const int64_t slots = (budget - 1024 - P.x_bytes - P.part_bytes) / P.slot_bytes;
        const int64_t want = std::min<int64_t>(L == kLevels - 1 ? 2 : 3, std::max<int64_t>(2, P.stages));
        if (slots >= want) P.level = L;
    }
    if (P.level >= 0) {
        P.xsmem = true;
    } else {
        const kq_status ps = plan_level(mats, n, ntok, ncta, 0, P);
        if (ps != KQ_OK) return ps;
        P.x_bytes = 0;
    }
    const int64_t fixed = 1024 + P.x_bytes + P.part_bytes + P.scr_bytes;
    P.nslot = std::min<int64_t>(kq::kMaxSlots, (budget - fixed) / P.slot_bytes);
    if (P.nslot < 2) return KQ_ERR_SHAPE;
    P.smem = fixed + P.nslot * P.slot_bytes;
    return KQ_OK;
}

bool tc_stream_preferred(const Plan &P) {
    if (P.tc_noct < 2) return true;
    for (int i = 0; i < P.n; ++i) {
        const Member &M = P.m[i];
        // CTAs of rows_q rows exist when rows_r < ncta, of rows_q + 1 when rows_r > 0
        const bool occurs[2] = {M.rows_r < M.ncta, M.rows_r > 0};
        for (int big = 0; big < 2; ++big) {
            if (!occurs[big] || M.ng[big] <= 1) continue;
            // groups of gq rows, and of gq + 1 when gr > 0: each must fill
            // four fifths of its 16-row tiles
            for (int hh = M.gq[big]; hh <= M.gq[big] + (M.gr[big] > 0 ? 1 : 0); ++hh) {
                const int tiles = (hh + 15) / 16;
                if (5 * hh < 4 * 16 * tiles) return false;
            }
        }
    }
    return true;
}

int stream_consumers(const Plan &P, const kq_mat *mats, int n) {
    bool tall = P.tc_noct == 0 && P.ntok == 1 && P.xsmem && P.stages >= 8;
    for (int i = 0; i < n; ++i) tall = tall && mats[i].fmt == KQ_Q6_K;
    return tall ? kq::kStreamConsumersTall : kq::kStreamConsumers;
}

int stream_rows_per_lane(const Plan &P, const kq_mat *mats, int n) {
    if (stream_consumers(P, mats, n) != kq::kStreamConsumersTall) return 2;
    for (int i = 0; i < n; ++i)
        if (P.m[i].whole) return 2;
    return 1;
}

}  // namespace kqplan

extern "C" int kq_plan_describe(const kq_mat *mats, int n, int ntok, int sms, int smem_optin,
                                int64_t *out, int cap) {
    if (!mats || !out || n < 1 || n > KQ_MAX_SET || ntok < 1 || ntok > KQ_MAX_NTOK || sms < 1)
        return -1;
    if (cap < KQ_PLAN_HEAD + n * KQ_PLAN_MEMBER) return -1;
    kqplan::Plan P;
    const int noct = ntok >= kq::kTcMinNtok ? (ntok + 7) / 8 : 0;
    if (noct == 0 && ntok > 8) return -1;
    const kq_status st = kqplan::plan_stream(mats, n, ntok, sms, smem_optin, &P, noct);
    int64_t *o = out;
    *o++ = st;
    *o++ = P.grid;
    *o++ = P.level;
    *o++ = P.xsmem ? 1 : 0;
    *o++ = P.x_bytes;
    *o++ = P.part_bytes;
    *o++ = P.slot_bytes;
    *o++ = P.nslot;
    *o++ = P.smem;
    *o++ = P.stages;
    *o++ = P.scr_bytes;
    *o++ = P.part_bufs;
    *o++ = st == KQ_OK && noct > 0 ? (kqplan::tc_stream_preferred(P) ? 1 : 0) : 0;
    *o++ = st == KQ_OK ? kqplan::stream_consumers(P, mats, n) : 0;
    *o++ = st == KQ_OK ? kqplan::stream_rows_per_lane(P, mats, n) : 0;
    for (int i = 0; i < n; ++i) {
        const kqplan::Member &M = P.m[i];
        const int64_t v[KQ_PLAN_MEMBER] = {M.ncta, M.cta_begin, M.rows_q, M.rows_r, M.ng[0],
                                           M.gq[0], M.gr[0], M.ng[1], M.gq[1], M.gr[1],
                                           M.rmax, M.kb, M.seg, M.hmax, M.nh, M.hs[0],
                                           M.hs[1], M.hs[2], M.hs[3], M.row_bytes,
                                           M.whole};
        for (int k = 0; k < KQ_PLAN_MEMBER; ++k) *o++ = v[k];
    }
    return 0;
}
