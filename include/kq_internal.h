/*
 * kq_internal.h -- introspection and test hooks of libkq.so.  Not part of
 * the matvec path: no call here touches a GPU or launches anything.
 */
#ifndef KQ_INTERNAL_H
#define KQ_INTERNAL_H

#include <stdint.h>

#include "kq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Entries of kq_plan_describe's output: KQ_PLAN_HEAD for the launch, then
 * KQ_PLAN_MEMBER per member. */
#define KQ_PLAN_HEAD 15
#define KQ_PLAN_MEMBER 21

/*
 * The streaming kernel's launch geometry for the set `mats` (n members,
 * ntok token columns in the launch: the dp4a launch for 1..3, the
 * tensor-core launch for 4..16; the library also runs a wide matrix at
 * 2..3 on the tensor cores, see kq.h) on a device with `sms` SMs and
 * `smem_optin` bytes of opt-in shared memory per CTA, as the library would
 * plan it.  Pure host arithmetic on the descriptors' shapes and formats
 * (their pointers are not read).
 *
 * out (host, at least KQ_PLAN_HEAD + n * KQ_PLAN_MEMBER int64 entries):
 *   [0] kq_status of the plan (KQ_ERR_SHAPE: the direct kernel would run)
 *   [1] grid  [2] level (-1: records in global memory)  [3] records in
 *   shared memory (0/1)  [4] x_bytes  [5] part_bytes  [6] slot_bytes
 *   [7] nslot  [8] dynamic shared memory  [9] stages of the largest CTA
 *   [10] bytes of the tensor-core units' scratch (0 for dp4a launches)
 *   [11] partial buffers (2; 1 for a tensor-core launch whose CTAs have
 *   one row group each)  [12] tensor-core launches: 1 if the library takes
 *   the streaming kernel for this plan under automatic kernel selection,
 *   0 if it takes the direct-load kernel (two octets of tokens and several
 *   row groups a CTA that fill less than four fifths of their 16-row
 *   tiles); 0 for dp4a launches and failed plans  [13] consumer warps of the
 *   streaming launch (12; 15 for one token column of Q6_K-only members
 *   with records in shared memory and 8 or more stages a CTA); 0 for
 *   failed plans  [14] rows of one lane-task in a dp4a launch (2; 1 in
 *   the 15-warp launch when no member is staged in whole rows); 0 for
 *   failed plans
 *   then per member: ncta, cta_begin, rows_q, rows_r, ng0, gq0, gr0, ng1,
 *   gq1, gr1, rmax, kb, seg, hmax, nh, hs0..hs3, row_bytes, whole (Q6_K
 *   stages of whole rows, one bulk copy each: 1; else 0).
 * Returns 0, or -1 for bad arguments (nothing written).
 */
int kq_plan_describe(const kq_mat *mats, int n, int ntok, int sms, int smem_optin,
                     int64_t *out, int cap);

/*
 * Test hook for failure reporting: the wall-time limit, in nanoseconds, of
 * every wait the streaming kernel makes on a shared-memory barrier (and of
 * its producer's wait for the input loads), for launches enqueued after
 * this call; 0 restores the default of 2 s.  Returns the previous setting
 * (0 = default).  Process-wide.
 *
 * A limit far below the time the weights take to arrive makes waits expire
 * on purpose.  The kernel then does what it does on a real expiry: the CTA
 * sets its abort flag and the device error word (kq_device_error reports
 * KQ_ERR_TIMEOUT), stops issuing copies, waits -- always with the default
 * limit -- for the copies it had issued, and writes NaN to the rows it had
 * not finished.  Nothing hangs or faults, and the next launch made with the
 * default limit computes normally.
 */
unsigned long long kq_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* KQ_INTERNAL_H */
