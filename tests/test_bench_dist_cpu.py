"""bench.py's multi-process logic on CPU (no GPU): the max-over-ranks timing
with a world-size-2 gloo group, the whole-job byte count, and the reference
arm under torchrun (rank 0 alone prints one line; every rank exits 0)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

torch = pytest.importorskip("torch")


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's "time": the job's time is the slowest rank's
        mine = [3.25, 7.5][rank]
        got = bench.max_over_ranks(mine, dist, "cpu")
        dist.barrier()
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2(tmp_path):
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert float((tmp_path / f"r{r}").read_text()) == 7.5


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(4.5, None) == 4.5


def test_job_value_counts_every_rank():
    # 1 GB per step, 10 steps, 2 ranks, 1 s: 20 GB/s for the job
    assert bench.job_gbs(1e9, 10, 2, 1000.0) == pytest.approx(20.0)
    assert bench.job_gbs(1e9, 10, 1, 1000.0) == pytest.approx(10.0)


def test_reference_arm_under_torchrun_world2():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "3", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
