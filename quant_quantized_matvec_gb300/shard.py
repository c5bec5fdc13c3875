"""Row-sharded matvec over several GPUs: each rank owns a contiguous range of
rows, x is replicated, and one all-gather assembles y.

"Chapter 13 - The QKV + gate matvec family", section 13.3: every output row
is an independent dot product of its own weight row with the shared input,
so a matrix splits by rows with no change to any row's arithmetic -- a
gathered y is bitwise the one-GPU result.  Splitting the columns instead
would need an all-reduce and would change the sum order, so it is not done.

Shard boundaries fall on whole rows, at multiples of the smallest row count
whose bytes are a multiple of 16, so that every shard's weights start on the
16-byte boundary the kernels require (Q4_K and Q5_K rows are multiples of 16
bytes; a Q6_K row of 6656 inputs is 5460 bytes, so Q6_K shards start at
multiples of 4 rows there).

This module is host logic and argument marshalling only: the per-rank matvec
is kq.matvec (the CUDA library) and the exchange is torch.distributed's
all-gather (NCCL on GPUs), of each rank's [ntok, pad_rows] block (shards
padded to the largest one); the caller's y receives the real rows.  No
library kernel reads another GPU's memory.
"""
from __future__ import annotations

import math

from . import synth

__all__ = ["row_align", "row_shards", "local_rows", "sharded_matvec"]


def row_align(fmt: int, cols: int) -> int:
    """Smallest number of rows whose bytes are a multiple of 16."""
    row_bytes = (cols // 256) * synth.BLOCK_BYTES[fmt]
    return 16 // math.gcd(row_bytes, 16)


def row_shards(fmt: int, rows: int, cols: int, world: int):
    """[(start, stop)] for each rank: contiguous, in rank order, covering
    0..rows once; every start a multiple of row_align(fmt, cols); sizes as
    equal as that alignment allows (a rank may get an empty range when rows
    are fewer than world * alignment)."""
    if world < 1 or rows < 1:
        raise ValueError("world and rows must be positive")
    a = row_align(fmt, cols)
    units = -(-rows // a)                      # aligned row units
    bounds = [min(rows, a * ((units * r) // world)) for r in range(world + 1)]
    bounds[-1] = rows
    return [(bounds[r], bounds[r + 1]) for r in range(world)]


def local_rows(W_full, fmt: int, rows: int, cols: int, rank: int, world: int):
    """This rank's weight rows (a view of a row-major uint8 matrix, flat or
    [rows, row_bytes]) and its (start, stop)."""
    start, stop = row_shards(fmt, rows, cols, world)[rank]
    row_bytes = (cols // 256) * synth.BLOCK_BYTES[fmt]
    flat = W_full.reshape(-1)
    return flat[start * row_bytes: stop * row_bytes], (start, stop)


def sharded_matvec(fmt, W_local, rows, cols, x, y, group=None, local_matvec=None):
    """y[t, :] = W x[t, :] with W split by rows over the ranks of `group`.

    W_local  this rank's rows (row_shards(fmt, rows, cols, world)[rank]),
             uint8 bytes, on this rank's device.
    x        [ntok, cols] f32, the same on every rank.
    y        [ntok, rows] f32, overwritten with the whole result on every
             rank.
    local_matvec(fmt, W_local, nrows, cols, x) -> [ntok, nrows]: the
             per-rank matvec; kq.matvec by default.
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    shards = row_shards(fmt, rows, cols, world)
    pad = max(b - a for a, b in shards)
    ntok = x.shape[0]
    if local_matvec is None:
        from . import matvec as local_matvec
    start, stop = shards[rank]
    part = torch.zeros((ntok, pad), dtype=torch.float32, device=y.device)
    if stop > start:
        part[:, :stop - start] = local_matvec(fmt, W_local, stop - start, cols, x)
    gathered = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(gathered, part, group=group)
    for r, (a, b) in enumerate(shards):
        if b > a:
            y[:, a:b] = gathered[r][:, :b - a]
    return y
