#!/usr/bin/env python3
"""Benchmark of the K-quant matvec on GB300: achieved HBM GB/s and us/call.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--ntok T]

A step is one pass of the whole hot path over one batch of synthetic input:
by default the Muse Glimmer QKV+gate concurrent set at ntok=1 (Q and gate
4096x6656 Q4_K, K and V 256x6656 Q6_K, one shared x) in ONE kq_matvec_set
launch.  Other workloads (--workload) time the single-matrix shapes, the
Q6_K+Q5_K grid-split pair, the LM head and the embedding lookup (embed_q4k:
--ntok token rows of a 202048x6656 Q4_K table per step, kq_dequant_rows).

Timing (ours): inputs resident in HBM; K steps replayed from CUDA graphs,
bracketed by CUDA events on the launching stream with a barrier and a device
synchronize on both sides; the weights rotate over enough copies that their
total exceeds three times the L2 size, so every step streams from HBM.
`value` = algorithmic bytes (weights + x once per distinct plane + y) of all
steps on all ranks / max-over-ranks elapsed time.  By default the calls run
with launch overlap on (kq_set_overlap: a call streams its weights while the
previous call finishes and reads x only after that call completes); the
same K steps with overlap off are timed too and reported as `serial`
(--no-overlap makes them the headline).  `replays` gives the median,
minimum and maximum us per call over the graph replays of the timed region.
`e2e` times the public Python API with x and y in pinned host memory: each
call copies its x in and writes its y back inside the timed region (weights
stay resident, as model weights do); the same steps with explicit copies
around device buffers are reported beside it.  Timed regions are preceded by
an untimed pre-warm (--prewarm-ms of graph replays) and a GPU sleep
(--head-start-ms), so that they measure steady state and not the host's
launch gap.  `cpu_baseline` times the CPU
oracle on a bounded sample, single-threaded and (`all_cores`) with the rows
split over every host core.

--impl reference times the CPU oracle itself (single thread), one pass over
the workload's matrices per step (2048 fresh random rows of any matrix above
64 MB), and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from quant_quantized_matvec_gb300 import synth  # noqa: E402

Q4_K, Q5_K, Q6_K = synth.Q4_K, synth.Q5_K, synth.Q6_K
METRIC = ("achieved HBM GB/s (% of GB300 peak) and us per K-quant matvec, "
          "ntok=1")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # HBM3e spec figure, for context only


# ----------------------------------------------------------------- workloads
def workload(name: str, ntok: int):
    """-> (members [(fmt, rows, cols, x_plane)], description)."""
    if name == "qkv_gate_set":
        return ([(Q4_K, 4096, 6656, 0), (Q6_K, 256, 6656, 0),
                 (Q6_K, 256, 6656, 0), (Q4_K, 4096, 6656, 0)],
                "Muse Glimmer QKV+gate concurrent set: Q,gate 4096x6656 Q4_K;"
                " K,V 256x6656 Q6_K; shared x; one kq_matvec_set launch")
    if name in ("q4k_4096", "q5k_4096", "q6k_4096"):
        fmt = {"q4k": Q4_K, "q5k": Q5_K, "q6k": Q6_K}[name[:3]]
        return ([(fmt, 4096, 6656, 0)],
                f"single {synth.FMT_NAMES[fmt]} 4096x6656 matvec")
    if name == "q4k_256":
        return ([(Q4_K, 256, 6656, 0)], "single Q4_K 256x6656 matvec")
    if name == "cat_q6k_q5k":
        return ([(Q6_K, 512, 2560, 0), (Q5_K, 512, 2560, 1)],
                "grid-split pair Q6_K + Q5_K 2560->512, separate x planes")
    if name == "lm_head_q6k":
        return ([(Q6_K, 202048, 6656, 0)], "LM head Q6_K 202048x6656")
    if name == "lm_head_q6k_slice":
        # the LM head's launch form (whole-row stages, 15 consumer warps) on
        # 260 rows a CTA: 216 MB, above L2, small enough for a many-pass ncu
        # capture
        return ([(Q6_K, 39520, 6656, 0)], "LM head Q6_K rows 0..39519 (39520x6656)")
    # further release shapes ("Chapter 6 - The kquant family on the
    # reference lane", Figure 6.6; n_in -> n_out is cols -> rows)
    if name == "ffn_gate_up_set":
        return ([(Q4_K, 19968, 6656, 0), (Q4_K, 19968, 6656, 0)],
                "FFN gate + up concurrent set: 2 x Q4_K 6656->19968, shared x")
    if name == "ffn_down_q4k":
        return ([(Q4_K, 6656, 19968, 0)], "FFN down Q4_K 19968->6656")
    if name == "ffn_down_q6k":
        return ([(Q6_K, 6656, 19968, 0)], "FFN down Q6_K 19968->6656")
    if name == "attn_output_q4k":
        return ([(Q4_K, 6656, 4096, 0)], "attention output Q4_K 4096->6656")
    if name == "lm_head_q5k":
        return ([(Q5_K, 202048, 6656, 0)], "LM head Q5_K 6656->202048")
    if name == "draft_kv_set":
        return ([(Q4_K, 1024, 6656, 0), (Q6_K, 1024, 6656, 0)],
                "draft k + v set: Q4_K and Q6_K 6656->1024, shared x")
    if name == "draft_fc_q4k":
        return ([(Q4_K, 6656, 33280, 0)], "draft fc Q4_K 33280->6656")
    if name == "embed_q4k":
        return ([(Q4_K, 202048, 6656, 0)],
                "embedding lookup: ntok token rows of a 202048x6656 Q4_K table "
                "gathered and dequantized to f32 (kq_dequant_rows)")
    raise SystemExit(f"unknown workload {name}")


def algorithmic_bytes(members, ntok) -> int:
    """Weights + each distinct x plane once + every y."""
    w = sum(rows * (cols // 256) * synth.BLOCK_BYTES[f]
            for f, rows, cols, _ in members)
    planes = {}
    for f, rows, cols, p in members:
        planes[p] = cols
    x = sum(4 * ntok * c for c in planes.values())
    y = sum(4 * ntok * rows for _, rows, _, _ in members)
    return w + x + y


def host_inputs(members, ntok, label):
    Ws = [synth.kquant_matrix(f, r, c, f"{label}/W{i}")
          for i, (f, r, c, _) in enumerate(members)]
    planes = {}
    for f, r, c, p in members:
        if p not in planes:
            planes[p] = synth.activations(ntok, c, f"{label}/x{p}")
    return Ws, planes


# ----------------------------------------------------------------- helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quant_quantized_matvec_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name, ntok):
    """DRAM bytes per launch from a committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(f"{workload_name}/ntok{ntok}")
        if e and e.get("kernel_source_hash") == kernel_source_hash():
            return int(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def props_clock_hz(props) -> float:
    """SM clock for converting a sleep length to cycles (the maximum clock,
    so a sleep is at least as long as asked)."""
    mhz = getattr(props, "clock_rate", 0) / 1e3 if getattr(props, "clock_rate", 0) else 2070.0
    return max(mhz, 2070.0) * 1e6


def max_over_ranks(value, dist, device=None):
    """The largest of every rank's value (a job takes as long as its slowest
    rank); `value` itself when the run is not distributed."""
    if not dist:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes, steps, world, ms):
    """Whole-job throughput: the bytes every rank processed over the job's
    time (the slowest rank's), in GB/s."""
    return step_bytes * steps * world / (ms * 1e-3) / 1e9


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv",
                                                 delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.seek(0)
        rows = [ln.split(",") for ln in self.f.read().splitlines() if ln]
        self.f.close()
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(members, Ws, planes, ntok, budget_s=10.0):
    """The oracle as it stands, single-threaded, on whole matrices of the
    workload (a row sample for matrices too large to finish in budget)."""
    import oracle
    oracle.build()
    done_bytes, t0, reps = 0, time.perf_counter(), 0
    rng = np.random.default_rng(0)
    sample_desc = None
    while True:
        for i, (f, r, c, p) in enumerate(members):
            bpr = (c // 256) * synth.BLOCK_BYTES[f]
            if r * bpr > 64 << 20:
                idx = np.sort(rng.choice(r, size=2048, replace=False))
                oracle.matvec(f, Ws[i], r, c, planes[p], row_idx=idx)
                done_bytes += len(idx) * bpr + 4 * ntok * (c + len(idx))
                sample_desc = "2048 random rows per pass"
            else:
                oracle.matvec(f, Ws[i], r, c, planes[p])
                done_bytes += r * bpr + 4 * ntok * (c + r)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    gbs = done_bytes / el / 1e9
    line = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": (sample_desc or
                       f"{reps} full pass(es) of the workload") +
            f", {el:.1f} s single-threaded (f32 dequant + f64 dots)"}
    line["all_cores"] = cpu_baseline_all_cores(members, Ws, planes, ntok,
                                               budget_s / 2)
    return line


def cpu_baseline_all_cores(members, Ws, planes, ntok, budget_s=5.0):
    """The same oracle calls spread over every host core: each thread takes
    a contiguous share of every matrix's rows (the C oracle releases the
    interpreter lock and keeps no shared state)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    jobs = []  # (matrix, row indices, bytes)
    sampled = False
    for i, (f, r, c, p) in enumerate(members):
        bpr = (c // 256) * synth.BLOCK_BYTES[f]
        if r * bpr > 64 << 20:
            rows = np.sort(rng.choice(r, size=2048 * cores, replace=False))
            sampled = True
        else:
            rows = np.arange(r)
        for part in np.array_split(rows, cores):
            if len(part):
                jobs.append((i, part, len(part) * bpr + 4 * ntok * (c + len(part))))

    def run(job):
        i, rows, nbytes = job
        f, r, c, p = members[i]
        oracle.matvec(f, Ws[i], r, c, planes[p], row_idx=rows)
        return nbytes

    done_bytes, reps = 0, 0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        t0 = time.perf_counter()
        while True:
            done_bytes += sum(ex.map(run, jobs))
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    return {"value": round(done_bytes / el / 1e9, 4), "unit": "GB/s",
            "cores": cores, "kind": "oracle",
            "sample": (f"{2048 * cores} random rows per large matrix"
                       if sampled else f"{reps} full pass(es) of the workload")
            + f", {el:.1f} s on {cores} threads, rows split evenly"}


# ----------------------------------------------------------------- ours
def run_ours(args, rank, world, dist):
    import torch

    import quant_quantized_matvec_gb300 as kq
    from quant_quantized_matvec_gb300 import build as kbuild
    kbuild.build()
    kq._binding.load()

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    members, desc = workload(args.workload, args.ntok)
    ntok = args.ntok
    Ws, planes = host_inputs(members, ntok, f"bench/{args.workload}")
    step_bytes = algorithmic_bytes(members, ntok)
    w_bytes = sum(W.nbytes for W in Ws)

    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or (126 << 20))
    copies = max(1, -(-3 * l2 // w_bytes)) if w_bytes < 3 * l2 else 1
    Wd = [[torch.from_numpy(W.reshape(-1)).to(dev) for W in Ws]]
    for _ in range(copies - 1):
        Wd.append([w.clone() for w in Wd[0]])
    xd = {p: torch.from_numpy(x).to(dev) for p, x in planes.items()}
    y_all = torch.empty(sum(ntok * r for _, r, _, _ in members),
                        dtype=torch.float32, device=dev)
    ys, off = [], 0
    for f, r, c, p in members:
        ys.append(y_all[off:off + ntok * r].view(ntok, r))
        off += ntok * r
    sets = []
    for cpy in Wd:
        mem = [(f, cpy[i], r, c, xd[p], ys[i])
               for i, (f, r, c, p) in enumerate(members)]
        sets.append((mem, kq.make_set(mem)))

    # the calls take their temporaries (tensor-core input fragments, staged
    # host inputs, global input records) from one preallocated workspace
    # (kq_matvec_set_ws) instead of stream-ordered allocations, so a step is
    # kernels only; calls on one stream may share it
    ws = torch.empty(max(kq.workspace_bytes(d, ntok) for _, d in sets),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def step(i):
        mem, d = sets[i % len(sets)]
        kq.matvec_set(mem, ntok=ntok, stream=stream, descriptors=d, workspace=ws)

    K = args.steps
    L = min(K, args.graph_len)
    head_cycles = int(args.head_start_ms * 1e-3 * props_clock_hz(props))

    def timed(overlap, sampler=None, stepfn=step, K=K):
        """K steps replayed from CUDA graphs of L steps, captured with the
        given launch-overlap setting; -> ms (max over ranks), wall s,
        (replays, remainder steps), µs per call of each main-graph replay,
        pre-warm ms.

        Steady state: before the timed region the main graph is replayed,
        untimed, for at least --prewarm-ms of wall time (clocks and caches
        settle, the launch path is warm), and a GPU sleep of --head-start-ms
        is queued just before the start event, so that the host has queued
        every timed replay before the GPU reaches that event: the timed
        region holds exactly K calls and no host launch gap."""
        kq.set_overlap(overlap)
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                stepfn(i)
        torch.cuda.synchronize()

        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    stepfn(i)
            return g

        L = min(K, args.graph_len)
        g_main = capture(L)
        reps, rem = K // L, K % L
        g_rem = capture(rem) if rem else None
        torch.cuda.synchronize()
        t_pre = time.perf_counter()
        with torch.cuda.stream(stream):
            while True:
                g_main.replay()
                if g_rem is not None:
                    g_rem.replay()
                torch.cuda.synchronize()
                if time.perf_counter() - t_pre >= args.prewarm_ms * 1e-3:
                    break
        prewarm_ms = (time.perf_counter() - t_pre) * 1e3
        if sampler:
            sampler.start()
            time.sleep(0.3)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        # one event after each replay of the main graph: per-replay times
        # for the median (recorded between replays, on the same stream)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(head_cycles)  # outside the timed region
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for r in range(reps):
                g_main.replay()
                evs[r].record(stream)
            if g_rem is not None:
                g_rem.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        if dist:
            dist.barrier()
        ms = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
        per_replay = [ev0.elapsed_time(evs[0])] + [
            evs[r - 1].elapsed_time(evs[r]) for r in range(1, reps)]
        return ms, wall, (reps, rem), [1e3 * t / L for t in per_replay], prewarm_ms

    overlap = not args.no_overlap
    ms_serial = timed(False)[0]
    # warm: the same calls on one weight copy, which stays in L2 when it fits
    Kw = min(K, 20000)
    ms_warm = (timed(overlap, stepfn=lambda i: step(0), K=Kw)[0]
               if copies > 1 else None)
    sampler = ClockSampler(dev.index)
    ms, wall, (reps, rem), per_replay, prewarm_ms = timed(overlap, sampler)
    per_replay = sorted(per_replay)
    clocks = sampler.stop()
    kernels = kq.last_kernels()
    launches_per_step = kq.last_launch_count()
    gbs = job_gbs(step_bytes, K, world, ms)
    us_per_step = ms * 1e3 / K

    # End to end through the public API, every step: the call takes x and y
    # in pinned host memory -- the library copies x in with a staging kernel
    # that the matvec overlaps, and the matvec writes y straight into host
    # memory.  The same steps with device buffers and explicit copies in and
    # out are reported beside it.
    x_host = {p: torch.from_numpy(x).pin_memory() for p, x in planes.items()}
    y_host = torch.empty(y_all.numel(), dtype=torch.float32).pin_memory()
    yh, off = [], 0
    for f, r, c, p in members:
        yh.append(y_host[off:off + ntok * r].view(ntok, r))
        off += ntok * r
    host_sets = []
    for cpy in Wd:
        mem = [(f, cpy[i], r, c, x_host[p], yh[i])
               for i, (f, r, c, p) in enumerate(members)]
        host_sets.append((mem, kq.make_set(mem)))
    Ke = min(K, args.e2e_steps)
    h2d = sum(x.numel() * 4 for x in x_host.values())
    d2h = y_host.numel() * 4
    kq.set_overlap(overlap)

    def e2e(host_y):
        """Ke steps through the public API, timed on the device; the host
        cost of issuing one step is measured separately, on the warm-up
        steps (wall clock of their loop, which never waits for the GPU).  A GPU sleep queued before the start
        event gives the host a head start of about the whole loop's issue
        time, so that the device timeline is the one a caller gets when it
        keeps the stream fed (as a serving loop or a captured graph does);
        -> (device ms, host µs per step)."""
        def one(i):
            if host_y:
                mem, d = host_sets[i % len(host_sets)]
                kq.matvec_set(mem, ntok=ntok, stream=stream, descriptors=d, workspace=ws)
            else:
                for p in xd:
                    xd[p].copy_(x_host[p], non_blocking=True)
                step(i)
                y_host.copy_(y_all, non_blocking=True)
        with torch.cuda.stream(stream):
            one(0)  # first call: one-time set-up (pointer lookups, tensor maps)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup)):
                one(i)
        host_us = (time.perf_counter() - t0) * 1e6 / max(3, args.warmup)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        lead_ms = min(200.0, 1.5 * host_us * Ke * 1e-3 + args.head_start_ms)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(lead_ms * 1e-3 * props_clock_hz(props)))
        e0.record(stream)
        with torch.cuda.stream(stream):
            for i in range(Ke):
                one(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1), dist, dev), host_us

    ems, host_us = e2e(True)
    y_direct = y_host.clone()
    ems_copy, host_us_copy = e2e(False)
    # the last step wrote the same outputs both ways
    e2e_same = bool(torch.equal(y_direct.view(torch.int32), y_host.view(torch.int32)))
    e2e_gbs = job_gbs(step_bytes, Ke, world, ems)

    peak, peak_kind = peaks()
    traffic = recorded_traffic(args.workload, ntok)
    line = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms / K, 6),
        "us_per_call": round(us_per_step, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded K-quant blocks, x ~ N(0,1))",
        "config": {
            "workload": args.workload, "description": desc,
            "ntok": ntok,
            "matrices": [f"{synth.FMT_NAMES[f]} {r}x{c}"
                         for f, r, c, _ in members],
            "bytes_per_step": step_bytes,
            "workspace_bytes": int(ws.numel()),
            "l2": (f"inputs rotate over {copies} weight copies "
                   f"({copies * w_bytes / 1e6:.0f} MB, L2 {l2 / 1e6:.0f} MB)"
                   if copies > 1 else
                   f"weights {w_bytes / 1e6:.0f} MB > 3x L2"),
            "timing": f"CUDA graphs of {L} calls, {reps} replays"
                      + (f" + {rem}" if rem else "") + ", events on stream"
                      + f"; untimed pre-warm of {prewarm_ms:.0f} ms of replays and a "
                        f"{args.head_start_ms:g} ms GPU head start before the timed region"
                      + ("; launch overlap on: a call's weights stream "
                         "while the previous call finishes, its x is read "
                         "after that call completes" if overlap else ""),
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
        },
        "gpu_launches": K * launches_per_step,
        "replays": {"n": len(per_replay), "calls_each": L,
                    "median_us_per_call": round(float(np.median(per_replay)), 3),
                    "min_us_per_call": round(per_replay[0], 3),
                    "max_us_per_call": round(per_replay[-1], 3),
                    "note": "per replay of the main graph inside the timed region (this rank)"},
        "launch_overlap": overlap,
        "prewarm_ms": round(prewarm_ms, 1),
        "warm_l2": ({"us_per_call": round(ms_warm * 1e3 / Kw, 3),
                     "value": round(job_gbs(step_bytes, Kw, world, ms_warm), 2),
                     "note": "warm, L2-resident: one weight copy reused every call "
                             "(not an HBM number)"} if ms_warm else None),
        "serial": {"us_per_call": round(ms_serial * 1e3 / K, 3),
                   "value": round(job_gbs(step_bytes, K, world, ms_serial), 2),
                   "note": "same steps with launch overlap off (each call "
                           "starts after the previous one completes)"},
        "roofline": {
            "bound": "hbm",
            "achieved": round(step_bytes / (ms * 1e-3 / K) / 1e9, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(step_bytes / (ms * 1e-3 / K) / 1e9 / peak, 4),
            "traffic": traffic,
            "peak_source": f"{peak_kind} HBM copy bandwidth",
            "frac_of_nominal": round(step_bytes / (ms * 1e-3 / K) / 1e9 / NOMINAL_HBM_GBS, 4),
            "kernel": ("kq_set_stream" if kernels["stream"] else "kq_set_direct")
                      + (" (tensor cores, after the fragment pass)" if kernels.get("tensor_cores") else ""),
            "launches_per_step": launches_per_step,
        },
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(ems * 1e3 / Ke, 3), "steps": Ke,
                "host_us_per_step": round(host_us, 3),
                "timing": "device time (CUDA events on the stream) of Ke calls "
                          "queued back to back; host_us_per_step is the host's "
                          "cost of issuing one call (Python + C ABI + launches)",
                "weights": "resident in HBM",
                "path": "x and y in pinned host memory, passed to the call: the "
                        "library copies x to the device with a staging kernel that "
                        "the matvec overlaps with its weight stream, and the matvec "
                        "writes y straight into host memory over the host link",
                "outputs_equal_copy_path": e2e_same,
                "copy_path": {"value": round(job_gbs(step_bytes, Ke, world, ems_copy), 2),
                              "us_per_step": round(ems_copy * 1e3 / Ke, 3),
                              "host_us_per_step": round(host_us_copy, 3),
                              "path": "x and y in device memory, with async copies "
                                      "from and to pinned host memory around each call"}},
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(members, Ws, planes, ntok,
                                            args.cpu_budget)
    return line


# ----------------------------------------------------------------- embedding
def run_embed(args, rank, world, dist):
    """The embedding lookup: ntok random token rows per step, gathered and
    dequantized by kq_dequant_rows; bytes = rows read + ids + f32 rows
    written."""
    import torch

    import quant_quantized_matvec_gb300 as kq
    from quant_quantized_matvec_gb300 import build as kbuild
    kbuild.build()
    kq._binding.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    (fmt, rows, cols, _), = workload(args.workload, args.ntok)[0]
    n = args.ntok
    W = synth.kquant_matrix(fmt, rows, cols, f"bench/{args.workload}/W")
    Wd = torch.from_numpy(W.reshape(-1)).to(dev)
    row_bytes = (cols // 256) * synth.BLOCK_BYTES[fmt]
    step_bytes = n * row_bytes + 4 * n + 4 * n * cols
    K = args.steps
    L = min(K, args.graph_len)
    rng = np.random.default_rng(1)
    ids_all = torch.from_numpy(
        rng.integers(0, rows, size=(L, n)).astype(np.int32)).to(dev)
    out = torch.empty((n, cols), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        kq.dequant_rows(fmt, Wd, rows, cols, ids_all[i % L], out=out,
                        stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(L):
            step(i)
    reps, rem = K // L, K % L
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            for i in range(rem):
                step(i)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    t_pre = time.perf_counter()
    with torch.cuda.stream(stream):
        while time.perf_counter() - t_pre < args.prewarm_ms * 1e-3:
            g.replay()
            torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(dev)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(args.head_start_ms * 1e-3 * props_clock_hz(props)))
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
        if g_rem is not None:
            g_rem.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    gbs = job_gbs(step_bytes, K, world, ms)
    # end to end: ids from pinned host memory, rows back to pinned host memory
    ids_host = torch.from_numpy(
        rng.integers(0, rows, size=n).astype(np.int32)).pin_memory()
    ids_dev = torch.empty(n, dtype=torch.int32, device=dev)
    out_host = torch.empty((n, cols), dtype=torch.float32).pin_memory()
    Ke = min(K, args.e2e_steps)
    torch.cuda.synchronize()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(Ke):
            ids_dev.copy_(ids_host, non_blocking=True)
            kq.dequant_rows(fmt, Wd, rows, cols, ids_dev, out=out, stream=stream)
            out_host.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ems = e0.elapsed_time(e1)
    peak, peak_kind = peaks()
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms / K, 6), "us_per_call": round(ms * 1e3 / K, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded Q4_K table, random token ids)",
        "config": {"workload": args.workload,
                   "description": workload(args.workload, n)[1],
                   "ntok": n, "bytes_per_step": step_bytes,
                   "l2": f"table {W.nbytes / 1e6:.0f} MB > 3x L2; random rows",
                   "timing": f"CUDA graphs of {L} calls, events on stream",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "gpu_launches": K,
        "roofline": {"bound": "hbm",
                     "achieved": round(step_bytes / (ms * 1e-3 / K) / 1e9, 2),
                     "peak": peak, "unit": "GB/s",
                     "frac": round(step_bytes / (ms * 1e-3 / K) / 1e9 / peak, 4),
                     "traffic": None,
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "kernel": "kq_rows_kernel", "launches_per_step": 1},
        "e2e": {"value": round(step_bytes * Ke / (ems * 1e-3) / 1e9, 2),
                "unit": "GB/s", "h2d_bytes_per_step": 4 * n,
                "d2h_bytes_per_step": 4 * n * cols,
                "us_per_step": round(ems * 1e3 / Ke, 3), "steps": Ke,
                "weights": "resident in HBM"},
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        t0, done, reps_c = time.perf_counter(), 0, 0
        while time.perf_counter() - t0 < args.cpu_budget:
            idx = rng.integers(0, rows, size=n).tolist()
            oracle.dequant_rows(fmt, W, cols, rows=idx)
            done += step_bytes
            reps_c += 1
        el = time.perf_counter() - t0
        line["cpu_baseline"] = {
            "value": round(done / el / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{reps_c} lookups of {n} random rows, {el:.1f} s "
                      "single-threaded (oracle dequantizer)"}
    return line


# ----------------------------------------------------------------- reference
def run_reference(args):
    """The CPU oracle as the reference arm: each step is one pass of the
    oracle over the whole workload, as cpu_baseline times it (a matrix above
    64 MB contributes 2048 rows drawn afresh every step, so that the sample
    does not stay in the host's caches)."""
    import oracle
    oracle.build()
    members, desc = workload(args.workload, args.ntok)
    ntok = args.ntok
    Ws, planes = host_inputs(members, ntok, f"bench/{args.workload}")
    embed = args.workload == "embed_q4k"
    rng = np.random.default_rng(1)
    sampled = []

    def step():
        if embed:  # the lookup itself: ntok random rows per step
            f, r, c, _ = members[0]
            oracle.dequant_rows(f, Ws[0], c, rows=rng.integers(0, r, size=ntok).tolist())
            return ntok * ((c // 256) * synth.BLOCK_BYTES[f] + 4 + 4 * c)
        nbytes = 0
        for i, (f, r, c, p) in enumerate(members):
            bpr = (c // 256) * synth.BLOCK_BYTES[f]
            if r * bpr > 64 << 20:
                idx = np.sort(rng.choice(r, size=2048, replace=False))
                oracle.matvec(f, Ws[i], r, c, planes[p], row_idx=idx)
                nbytes += len(idx) * bpr + 4 * ntok * (c + len(idx))
                sampled.append(i)
            else:
                oracle.matvec(f, Ws[i], r, c, planes[p])
                nbytes += r * bpr + 4 * ntok * (c + r)
        return nbytes

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    total = 0
    for _ in range(args.steps):
        total += step()
    el = time.perf_counter() - t0
    gbs = total / el / 1e9
    sample = ("ntok random token rows per step" if embed else
              "one pass over every matrix of the workload per step"
              + (" (2048 fresh random rows of each matrix above 64 MB)" if sampled else "")) \
        + f", {el:.1f} s single-threaded oracle (f32 dequant + f64 dots)"
    return {
        "metric": METRIC, "impl": "reference",
        "value": round(gbs, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded K-quant blocks)",
        "config": {"workload": args.workload, "description": desc,
                   "ntok": ntok},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qkv_gate_set")
    ap.add_argument("--ntok", type=int, default=1)
    ap.add_argument("--graph-len", type=int, default=2000)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--prewarm-ms", type=float, default=300.0,
                    help="untimed replays of the main graph before each timed region")
    ap.add_argument("--head-start-ms", type=float, default=2.0,
                    help="GPU sleep queued before the start event (host head start)")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overlap", action="store_true",
                    help="headline with launch overlap off")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
        dist = tdist
    if args.workload == "embed_q4k":
        line = run_embed(args, rank, world, dist)
    else:
        line = run_ours(args, rank, world, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
