// kq_plan.h -- launch geometry of the streaming kernel (host only).
//
// For a validated set: how many CTAs each member gets, how its rows split
// into row groups, the stage shape [h rows][kb blocks], the ring of
// shared-memory slots, and whether the input records fit in shared memory.
// Pure arithmetic on the shapes and two device facts (SM count, opt-in
// shared memory per CTA); kq_api.cu turns a plan into kernel parameters
// and tensor maps, and kq_plan_describe (kq_internal.h) exposes it to the
// host tests.
#pragma once

#include <stdint.h>

#include "kq.h"

namespace kqplan {

constexpr int kMaxHeights = 4;  // distinct row-group heights per member

struct Member {
    int ncta = 0, cta_begin = 0;
    int rows_q = 0, rows_r = 0;       // rows / ncta, rows % ncta
    int ng[2] = {}, gq[2] = {}, gr[2] = {};  // groups of CTAs with rows_q (+1) rows
    int rmax = 0;                     // rows per group at most
    int kb = 0;                       // blocks per stage row
    int seg = 0;                      // Q6_K: bytes between row segments in a slot
    int whole = 0;                    // Q6_K: stages of whole rows (one copy each)
    int nh = 0, hs[kMaxHeights] = {}; // group heights that occur
    int hmax = 0;
    int64_t row_bytes = 0;
};

struct Plan {
    int n = 0, ntok = 0, grid = 0;
    int level = -1;        // geometry level taken (records in global: level 0 geometry)
    bool xsmem = false;    // input records in shared memory
    int64_t x_bytes = 0, part_bytes = 0, slot_bytes = 0, nslot = 0, stages = 0;
    int part_bufs = 2;      // partial buffers (1 when no CTA has a second row group)
    int64_t scr_bytes = 0;  // tensor-core launches: the consumer warps' unit scratch
    int tc_noct = 0;        // tensor-core launches: octets of tokens (0: dp4a launch)
    int64_t smem = 0;      // dynamic shared memory of the launch
    Member m[KQ_MAX_SET];
};

// Consumer cost per weight byte of Q6_K relative to Q4_K, in sixteenths
// (measured: the Q6_K block loop spends more instructions per byte).
constexpr int64_t kCostQ6 = 32;

// The plan of one launch of `mats` (validated, 1..KQ_MAX_SET members).
// dp4a launches: ntok 1..8, records in shared memory when they fit.
// Tensor-core launches (tc_noct = 1 or 2 octets of tokens, ntok up to
// 8 * tc_noct): records in global memory, partials for 8 * tc_noct token
// columns (one buffer when no CTA has a second row group), and one unit
// scratch per consumer warp.  KQ_ERR_SHAPE when no geometry fits (the
// caller then uses the direct-load kernel).
// Tensor-core launches with two octets of tokens (9..16 columns): whether
// the streaming kernel is expected to beat the direct-load kernel on this
// plan.  It is where each CTA's rows form one group, or where every group
// fills at least four fifths of its 16-row tiles; with several thinner
// groups a CTA (each summed by one warp while the others go on, with twice
// the partials of one octet, and fewer weight slots beside them) the direct
// kernel's full 16-row tiles were faster on GB300: 6656x6656 Q4_K 26.7 vs
// 32.5 us, Q6_K 28.0 vs 39.0, FFN down 6656x19968 Q6_K 122.6 vs 150.5, while
// 4096x6656, 3072x6656 (one group) and 8192x6656 Q5_K (groups of 26-27
// rows) ran faster streamed.  One octet: always true.
bool tc_stream_preferred(const Plan &P);

// Consumer warps of a dp4a streaming launch: kq::kStreamConsumersTall (15)
// for one token column of Q6_K-only members with records in shared memory
// and 8 or more stages a CTA (the Q6_K LM head, FFN down), else
// kq::kStreamConsumers (12).  Tensor-core launches: kq::kStreamConsumers.
int stream_consumers(const Plan &P, const kq_mat *mats, int n);

// Rows of one lane-task in a dp4a streaming launch: 1 for the 15-warp
// launch of tall Q6_K sets when no member is staged in whole rows (FFN
// down: 34.4 against 36.4 us with 2; with whole-row stages, the LM head,
// one row a task took 254 against 207 us), else 2.  Tensor-core launches:
// 2 (unused).  A task count h x kb stays below 2^12 either way: segment
// stages hold at most 32 rows of at most 9 Q6_K blocks.
int stream_rows_per_lane(const Plan &P, const kq_mat *mats, int n);

kq_status plan_stream(const kq_mat *mats, int n, int ntok, int sms, int smem_optin, Plan *out,
                      int tc_noct = 0);

}  // namespace kqplan
