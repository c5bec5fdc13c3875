"""The streaming kernel's launch plan (kq_plan.cu), checked on the host with
no GPU through kq_plan_describe (include/kq_internal.h): for many shapes,
formats, set compositions and ntok, the plan must fit the device, cover
every row exactly once, keep stage task counts in the kernel's range and
size Q6_K row segments for their misalignment."""
import ctypes
import itertools

import numpy as np
import pytest

from quant_quantized_matvec_gb300 import _binding

HEAD, MEMBER = 15, 21
TC_MIN = 4                      # ntok from which the tensor-core path runs
TC_SCR = 12 * 16 * 28 * 4       # its unit scratch: 12 consumer warps, one 16-row tile
# ... and two tiles where units span both tiles of a group (ntok 9..16, groups of 17+ rows)
SMS, SMEM = 152, 232448          # GB300: SMs, opt-in shared memory per CTA
BB = {12: 144, 13: 176, 14: 210}
REC = {12: 832, 13: 832, 14: 1056}
OK, SHAPE = 0, 2


def plan(members, ntok, sms=SMS, smem=SMEM):
    lib = _binding.load()
    arr = (_binding.KqMat * len(members))()
    for i, (fmt, rows, cols) in enumerate(members):
        arr[i].fmt, arr[i].rows, arr[i].cols = fmt, rows, cols
        arr[i].W = arr[i].x = arr[i].y = 16 << 20  # never read
    out = (ctypes.c_int64 * (HEAD + MEMBER * len(members)))()
    assert lib.kq_plan_describe(arr, len(members), ntok, sms, smem, out, len(out)) == 0
    o = list(out)
    head = dict(zip(["status", "grid", "level", "xsmem", "x_bytes", "part_bytes",
                     "slot_bytes", "nslot", "smem", "stages", "scr_bytes", "part_bufs",
                     "tc_stream", "ncw", "rpt"],
                    o[:HEAD]))
    keys = ["ncta", "cta_begin", "rows_q", "rows_r", "ng0", "gq0", "gr0", "ng1", "gq1",
            "gr1", "rmax", "kb", "seg", "hmax", "nh", "hs0", "hs1", "hs2", "hs3", "row_bytes",
            "whole"]
    mem = [dict(zip(keys, o[HEAD + MEMBER * i: HEAD + MEMBER * (i + 1)]))
           for i in range(len(members))]
    return head, mem


def check(members, ntok, sms=SMS, smem=SMEM):
    h, mem = plan(members, ntok, sms, smem)
    if h["status"] != OK:
        assert h["status"] == SHAPE
        return h, mem
    # the grid: every member gets CTAs, at most one per row, in order; one
    # wave of one CTA per SM unless there are more members than SMs (CTAs
    # never wait on one another, so a second wave is only slower)
    assert 1 <= h["grid"] <= max(sms, len(members))
    begin = 0
    for (fmt, rows, cols), m in zip(members, mem):
        assert m["cta_begin"] == begin and 1 <= m["ncta"] <= rows
        begin += m["ncta"]
        # every row once: ncta CTAs of rows_q or rows_q + 1 rows
        assert m["rows_q"] * m["ncta"] + m["rows_r"] == rows and 0 <= m["rows_r"] < m["ncta"]
        nb = cols // 256
        assert m["row_bytes"] == nb * BB[fmt]
        for big in (0, 1):
            nn = m["rows_q"] + big
            ng, gq, gr = m[f"ng{big}"], m[f"gq{big}"], m[f"gr{big}"]
            # CTAs of rows_q + big rows exist only if rows_r > 0 (big) or
            # rows_r < ncta (not big)
            if nn == 0 or (big and m["rows_r"] == 0) or (not big and m["rows_r"] == m["ncta"]):
                continue
            assert ng * gq + gr == nn and 0 <= gr < ng
            assert gq + (1 if gr else 0) <= m["rmax"] <= 32
            assert gq + (1 if gr else 0) <= m["hmax"]
        heights = [m[f"hs{j}"] for j in range(m["nh"])]
        assert 1 <= m["nh"] <= 4 and max(heights) == m["hmax"]
        # partials of a group fit 64 KiB (tensor-core launches keep them
        # for 8 or 16 token columns)
        ntp = 8 * ((ntok + 7) // 8) if ntok >= TC_MIN else ntok
        # rows of the partials are nb x ntp + 1 floats (an odd stride)
        assert m["hmax"] * (nb * ntp + 1) * 4 <= 64 * 1024
        # stage rows: at most 2048 bytes (whole Q6_K rows: up to 8 KB),
        # tasks below 2^12
        assert ((m["hmax"] + 1) // 2) * m["kb"] < 4096
        # whole Q6_K rows only in dp4a launches of rows up to 8 KB
        assert not m["whole"] or (fmt == 14 and m["row_bytes"] <= 8192 and ntok < TC_MIN)
        if m["whole"]:
            # consecutive whole rows, one copy from the 16-byte boundary at
            # or below the first row to the one at or above the last byte
            assert m["kb"] == nb and m["seg"] == m["row_bytes"]
            wpart = m["hmax"] * m["row_bytes"] + 30
        elif fmt == 14:
            assert 1 <= m["kb"] <= nb and m["kb"] * BB[fmt] <= 2048
            # a segment holds kb blocks plus up to 14 bytes of misalignment
            # at each end, and is an odd number of 16-byte units
            assert m["seg"] >= m["kb"] * 210 + 28 and m["seg"] % 16 == 0 and (m["seg"] // 16) % 2 == 1
            wpart = m["hmax"] * m["seg"]
        else:
            assert 1 <= m["kb"] <= nb and m["kb"] * BB[fmt] <= 2048
            assert m["seg"] == 0
            assert (m["kb"] * BB[fmt]) % 8 == 0  # tensor-map box rows in u64
            wpart = m["hmax"] * m["kb"] * BB[fmt]
        assert h["slot_bytes"] >= wpart
        # two partial buffers unless no CTA has a second row group
        occurs = [m["rows_r"] < m["ncta"], m["rows_r"] > 0]
        if any(m[f"ng{big}"] > 1 for big in (0, 1) if occurs[big]):
            assert h["part_bufs"] == 2
        assert h["part_bufs"] in (1, 2) and (h["part_bufs"] == 2 or ntok >= TC_MIN)
        assert h["part_bytes"] >= h["part_bufs"] * m["hmax"] * (nb * ntp + 1) * 4
        if h["xsmem"]:
            assert h["x_bytes"] >= ntok * nb * REC[fmt]
    assert begin == h["grid"]
    # shared memory: records, partials and at least two slots within the opt-in
    assert h["nslot"] >= 2 and h["nslot"] <= 32
    assert h["smem"] == (1024 + h["x_bytes"] + h["part_bytes"] + h["scr_bytes"]
                         + h["nslot"] * h["slot_bytes"])
    # tensor-core launches: records in global memory, the units' scratch
    if ntok >= TC_MIN:
        tall = max(m["hmax"] for m in mem) > 16  # units of two tiles
        assert not h["xsmem"] and h["scr_bytes"] == TC_SCR * (2 if ntok > 8 and tall else 1)
    else:
        assert h["scr_bytes"] == 0
    assert h["smem"] <= smem - 1024
    if not h["xsmem"]:
        assert h["x_bytes"] == 0 and h["level"] == -1
    # routing under automatic kernel selection: one octet of tokens always
    # streams; with two, several row groups a CTA must each fill 4/5 of
    # their 16-row tiles
    if ntok < TC_MIN:
        assert h["tc_stream"] == 0
    elif ntok <= 8:
        assert h["tc_stream"] == 1
    else:
        fills = []
        for m in mem:
            occurs = [m["rows_r"] < m["ncta"], m["rows_r"] > 0]
            for big in (0, 1):
                if occurs[big] and m[f"ng{big}"] > 1:
                    q, r = m[f"gq{big}"], m[f"gr{big}"]
                    fills += [hh / (16 * -(-hh // 16)) for hh in ([q, q + 1] if r else [q])]
        assert h["tc_stream"] == int(all(f >= 0.8 for f in fills))
    # consumer warps: 15 only for one column of Q6_K-only sets with records
    # in shared memory and 8 or more stages a CTA; one row a lane-task only
    # there, and only without whole-row stages
    tall = (ntok == 1 and h["xsmem"] == 1 and h["stages"] >= 8
            and all(fmt == 14 for fmt, _, _ in members))
    assert h["ncw"] == (15 if tall else 12)
    one_row = tall and not any(m["whole"] for m in mem)
    assert h["rpt"] == (1 if one_row else 2)
    if one_row:
        assert all(m["hmax"] * m["kb"] < 4096 for m in mem)
    return h, mem


def test_qkv_gate_set_plan_matches_its_profile():
    """The QKV+gate set: 152 CTAs, records in shared memory, and the
    dynamic shared memory the committed ncu capture shows (215,168 B)."""
    qkv = [(12, 4096, 6656), (14, 256, 6656), (14, 256, 6656), (12, 4096, 6656)]
    h, mem = check(qkv, 1)
    assert h["status"] == OK and h["grid"] == 152 and h["xsmem"] == 1 and h["level"] == 0
    assert h["smem"] == 215168
    # Q6_K members get more CTAs per byte than Q4_K (cost weighting)
    q4_share = mem[0]["ncta"] / (4096 * 26 * 144)
    q6_share = mem[1]["ncta"] / (256 * 26 * 210)
    assert q6_share > q4_share


@pytest.mark.parametrize("fmt", [12, 13, 14])
@pytest.mark.parametrize("ntok", [1, 2, 3, 5, 8, 16])
def test_single_matrices(fmt, ntok):
    for rows, cols in itertools.product([1, 2, 31, 152, 153, 1000, 4096, 65536, 202048],
                                        [256, 768, 2560, 6656, 19968, 33280]):
        check([(fmt, rows, cols)], ntok)


def test_random_sets():
    rng = np.random.default_rng(5)
    planned = 0
    for _ in range(400):
        n = int(rng.integers(1, 17))
        ntok = int(rng.integers(1, 17))
        members = [(int(rng.choice([12, 13, 14])), int(rng.integers(1, 5000)),
                    256 * int(rng.choice([1, 3, 10, 26, 78]))) for _ in range(n)]
        h, _ = check(members, ntok)
        planned += h["status"] == OK
    # the rest fall back to the direct kernel: mostly wide matrices at
    # 9..16 tensor-core columns, whose partials leave no room for two slots
    assert planned > 150


@pytest.mark.parametrize("fmt,rows,cols,ntok,stream", [
    (12, 4096, 6656, 16, 1),   # one 26-27 row group a CTA
    (12, 3072, 6656, 16, 1),   # one 20-21 row group
    (13, 8192, 6656, 16, 1),   # groups of 26-27 rows: 4/5 of two tiles
    (12, 6656, 6656, 16, 0),   # groups of 21-22 rows
    (12, 6656, 4096, 12, 0),
    (14, 6656, 19968, 16, 0),  # groups of 10-11 rows
    (12, 5120, 6656, 16, 0),   # groups of 16 and 17 rows
    (12, 6656, 6656, 8, 1),    # one octet
])
def test_two_octet_launches_pick_the_kernel_measured_faster(fmt, rows, cols, ntok, stream):
    """Which kernel the library takes for a tensor-core launch it can
    stream (kq_plan.h, tc_stream_preferred: the streaming and direct-load
    kernels timed on GB300 for each of these shapes)."""
    h, _ = check([(fmt, rows, cols)], ntok)
    assert h["status"] == OK and h["tc_stream"] == stream


def test_more_members_than_sms_and_small_devices():
    check([(12, 64, 512)] * 16, 1, sms=8)
    check([(14, 3, 6656), (12, 5000, 6656)], 4, sms=16, smem=101376)


def test_shapes_the_stream_kernel_cannot_stage():
    """Partials of one row beyond 64 KiB (cols 2^20 at ntok 8) leave no
    geometry: the direct kernel runs instead."""
    h, _ = plan([(12, 64, 1 << 20)], 8)
    assert h["status"] == SHAPE


def test_plan_is_deterministic():
    members = [(12, 4096, 6656), (14, 256, 6656), (13, 777, 2560)]
    assert plan(members, 3) == plan(members, 3)


@pytest.mark.parametrize("members,ntok,ncw,rpt", [
    ([(14, 202048, 6656)], 1, 15, 2),                # Q6_K LM head (whole rows)
    ([(14, 39520, 6656)], 1, 15, 2),                 # its 39520-row slice
    ([(14, 6656, 19968)], 1, 15, 1),                 # Q6_K FFN down (segments)
    ([(14, 4096, 17920)], 1, 15, 1),
    ([(14, 15200, 2560)], 1, 15, 1),
    ([(14, 202048, 6656)], 2, 12, 2),                # two token columns
    ([(12, 202048, 6656)], 1, 12, 2),                # Q4_K LM head
    ([(12, 4096, 6656), (14, 256, 6656)], 1, 12, 2),  # mixed set
    ([(14, 4096, 6656)], 1, 12, 2),                  # 3 stages a CTA
    ([(14, 256, 6656)], 1, 12, 2),                   # one stage a CTA
    ([(14, 202048, 6656)], 8, 12, 2),                # tensor-core launch
])
def test_consumer_warps_and_task_rows(members, ntok, ncw, rpt):
    """Consumer warps of the launch (kq_plan.h, stream_consumers): 15 only
    for one token column of Q6_K-only sets with records in shared memory
    and 8 or more stages a CTA, else 12; tensor-core launches always 12.
    Rows a lane-task (stream_rows_per_lane): 1 only in that 15-warp launch
    when no member is staged in whole rows."""
    h, mem = plan(members, ntok)
    assert h["status"] == OK and h["ncw"] == ncw and h["rpt"] == rpt
    if ncw == 15:
        assert h["xsmem"] == 1 and h["stages"] >= 8
        assert rpt == (1 if not any(m["whole"] for m in mem) else 2)
    if rpt == 1:
        # one row a task: a stage's tasks are h x kb, below 2^12
        assert all(m["hmax"] * m["kb"] < 4096 for m in mem)


@pytest.mark.parametrize("ntok", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("name", ["qkv_gate_set", "q4k_4096", "q5k_4096", "q6k_4096",
                                  "q4k_256", "cat_q6k_q5k", "lm_head_q6k",
                                  "lm_head_q6k_slice", "ffn_gate_up_set", "ffn_down_q4k",
                                  "ffn_down_q6k", "attn_output_q4k", "lm_head_q5k",
                                  "draft_kv_set", "draft_fc_q4k"])
def test_bench_workloads_plan(name, ntok):
    """Every matvec workload the benchmark times plans a valid streaming
    launch on a GB300 (the checks of `check`) at ntok up to 8; at 16,
    where partials for 16 token columns leave the ring no room on some
    shapes (the QKV set, the LM heads, FFN gate+up), the plan reports
    KQ_ERR_SHAPE and the direct-load kernel runs, as it does when
    automatic selection prefers it."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    members, _ = bench.workload(name, ntok)
    h, _ = check([(f, r, c) for f, r, c, _ in members], ntok)
    assert h["status"] == OK or (ntok > 8 and h["status"] == SHAPE), (name, ntok)

