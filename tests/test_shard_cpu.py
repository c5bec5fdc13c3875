"""The row-sharded matvec (quant_quantized_matvec_gb300/shard.py) on CPU:
the row partition covers every row once with 16-byte-aligned shard starts,
and a world-size-2 gloo group that gathers per-rank results reproduces the
one-process result bit for bit.  The CPU oracle stands in for the per-rank
CUDA matvec (the exchange and the bookkeeping are what is under test; rows
are independent dot products, so a row's value does not depend on the
shard it falls in)."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from quant_quantized_matvec_gb300 import shard, synth  # noqa: E402

BB = {12: 144, 13: 176, 14: 210}


@pytest.mark.parametrize("fmt", [12, 13, 14])
def test_row_shards_cover_every_row_once_aligned(fmt):
    for cols in (256, 2560, 6656, 19968):
        rb = (cols // 256) * BB[fmt]
        a = shard.row_align(fmt, cols)
        assert (a * rb) % 16 == 0 and all((k * rb) % 16 for k in range(1, a))
        for rows in (1, 3, 4, 37, 256, 4096, 6656, 202048):
            for world in (1, 2, 3, 4, 8):
                sh = shard.row_shards(fmt, rows, cols, world)
                assert len(sh) == world and sh[0][0] == 0 and sh[-1][1] == rows
                for (a0, b0), (a1, b1) in zip(sh, sh[1:]):
                    assert b0 == a1
                for s0, s1 in sh:
                    assert 0 <= s0 <= s1 <= rows
                    assert (s0 * rb) % 16 == 0 or s0 == rows
                sizes = [s1 - s0 for s0, s1 in sh]
                if rows >= world * a:
                    assert max(sizes) - min(sizes) <= a


def test_q6k_rows_of_6656_shard_on_multiples_of_four():
    assert shard.row_align(14, 6656) == 4          # 5460-byte rows
    assert shard.row_align(12, 6656) == 1          # 3744-byte rows
    assert shard.row_shards(14, 37, 6656, 2) == [(0, 20), (20, 37)]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_matvec(fmt, W_local, nrows, cols, x):
    y, _ = oracle.matvec(fmt, np.ascontiguousarray(W_local.numpy()).reshape(nrows, -1),
                         nrows, cols, x.numpy())
    return torch.from_numpy(y.astype(np.float32))


def _rank_main(rank, world, port, cases, outdir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        for i, (fmt, rows, cols, ntok) in enumerate(cases):
            W = synth.kquant_matrix(fmt, rows, cols, f"shard/{i}/W")
            x = torch.from_numpy(synth.activations(ntok, cols, f"shard/{i}/x"))
            W_local, _ = shard.local_rows(torch.from_numpy(W.reshape(-1)), fmt, rows, cols,
                                          rank, world)
            y = torch.full((ntok, rows), float("nan"))
            shard.sharded_matvec(fmt, W_local, rows, cols, x, y,
                                 local_matvec=_oracle_matvec)
            np.save(os.path.join(outdir, f"y{i}_r{rank}.npy"), y.numpy())
    finally:
        dist.destroy_process_group()


def test_sharded_matvec_world2_gloo_equals_one_process(tmp_path):
    import torch.multiprocessing as mp
    cases = [(14, 37, 6656, 1), (12, 300, 2560, 2), (13, 5, 1024, 3)]
    mp.spawn(_rank_main, args=(2, _free_port(), cases, str(tmp_path)), nprocs=2, join=True)
    for i, (fmt, rows, cols, ntok) in enumerate(cases):
        W = synth.kquant_matrix(fmt, rows, cols, f"shard/{i}/W")
        x = synth.activations(ntok, cols, f"shard/{i}/x")
        y_one = oracle.matvec(fmt, W, rows, cols, x)[0].astype(np.float32)
        for r in range(2):
            y = np.load(tmp_path / f"y{i}_r{r}.npy")
            assert np.array_equal(y.view(np.uint32), y_one.view(np.uint32)), (i, r)
