"""The row-sharded matvec on the GPU (one GPU in this run).  Shards computed
by the CUDA kernels from row ranges of the device weights -- each a view
starting on a 16-byte boundary -- and put back together are bitwise the
whole matrix's result, for every world size the partition is asked for;
and sharded_matvec through a one-rank NCCL group equals kq.matvec."""
import os
import socket

import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402
from quant_quantized_matvec_gb300 import shard  # noqa: E402


@pytest.mark.parametrize("fmt", [kq.Q4_K, kq.Q5_K, kq.Q6_K])
@pytest.mark.parametrize("rows,cols,ntok", [(37, 6656, 1), (4096, 6656, 2), (300, 2560, 3)])
def test_shards_reassemble_bitwise(fmt, rows, cols, ntok):
    W, x = C.case(fmt, rows, cols, ntok, f"shardgpu/{fmt}/{rows}")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    y_full = kq.matvec(fmt, Wd, rows, cols, xd)
    for world in (2, 3, 4, 8):
        y = torch.full((ntok, rows), float("nan"), device="cuda")
        for rank in range(world):
            W_local, (a, b) = shard.local_rows(Wd, fmt, rows, cols, rank, world)
            if b > a:
                assert W_local.data_ptr() % 16 == 0
                y[:, a:b] = kq.matvec(fmt, W_local, b - a, cols, xd)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y_full.view(torch.int32)), world
    C.check(fmt, W, rows, cols, x, y_full.cpu().numpy(), what="unsharded")


def test_sharded_matvec_one_rank_nccl_group():
    import torch.distributed as dist
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    if not dist.is_nccl_available():
        pytest.skip("no NCCL in this torch")
    store = dist.TCPStore("127.0.0.1", port, 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    try:
        fmt, rows, cols, ntok = kq.Q6_K, 1000, 6656, 2
        W, x = C.case(fmt, rows, cols, ntok, "shardgpu/nccl")
        Wd, xd = C.to_dev(W), C.to_dev(x)
        W_local, _ = shard.local_rows(Wd, fmt, rows, cols, 0, 1)
        y = torch.empty((ntok, rows), device="cuda")
        shard.sharded_matvec(fmt, W_local, rows, cols, xd, y)
        y_ref = kq.matvec(fmt, Wd, rows, cols, xd)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y_ref.view(torch.int32))
    finally:
        dist.destroy_process_group()
