"""Seeded random cases through the C ABI: random formats, row counts (ragged,
tiny and large), cols (odd and even block counts), ntok 1..16, sets of
mixed members that share x or have their own, and outputs in device or
pinned host memory.  Every output is checked against the oracle at the
contract tolerance, and every set member bitwise against a separate call."""
import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402

FMTS = (kq.Q4_K, kq.Q5_K, kq.Q6_K)
NCASES = 24


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    ntok = int(rng.choice([1, 1, 1, 2, 3, 4, 5, 6, 7, 8, 11, 16]))
    nb = int(rng.choice([1, 2, 3, 5, 7, 10, 13, 18, 26, 37]))
    shared = bool(rng.integers(0, 2))
    n = int(rng.integers(1, 5))
    members = []
    for m in range(n):
        fmt = int(rng.choice(FMTS))
        rows = int(rng.choice([1, 2, 15, 16, 17, 31, 33, 64, 97, 255, 513, 1200]))
        mnb = nb if shared else int(rng.choice([1, 4, 9, 26]))
        members.append((fmt, rows, 256 * mnb))
    host_y = bool(rng.integers(0, 4) == 0)
    return ntok, shared, members, host_y


@pytest.mark.parametrize("seed", range(NCASES))
def test_random_set(seed):
    ntok, shared, members, host_y = draw(seed)
    xs, planes = [], {}
    descs, checks = [], []
    for i, (fmt, rows, cols) in enumerate(members):
        key = cols if shared else i
        if key not in planes:
            x = C.case(kq.Q4_K, 1, cols, ntok, f"fuzz/{seed}/x{key}")[1]
            planes[key] = (x, C.to_dev(x))
        x, xd = planes[key]
        W = C.case(fmt, rows, cols, 1, f"fuzz/{seed}/W{i}")[0]
        Wd = C.to_dev(W)
        if host_y:
            y = torch.full((ntok, rows), float("nan"), dtype=torch.float32).pin_memory()
        else:
            y = C.Guarded(ntok, rows)
        descs.append((fmt, Wd, rows, cols, xd, y if host_y else y.y))
        checks.append((fmt, W, rows, cols, x, y))
    kq.matvec_set(descs, ntok=ntok)
    torch.cuda.synchronize()
    for (fmt, W, rows, cols, x, y), (_, Wd, _, _, xd, _) in zip(checks, descs):
        got = y.numpy() if host_y else y.host()
        C.check(fmt, W, rows, cols, x, got, what=f"seed {seed} fmt {fmt} {rows}x{cols} ntok {ntok}")
        alone = C.Guarded(ntok, rows)
        kq.matvec(fmt, Wd, rows, cols, xd, y=alone.y)
        torch.cuda.synchronize()
        assert np.array_equal(np.ascontiguousarray(got).view(np.uint32),
                              alone.host().view(np.uint32)), f"seed {seed}: set != separate"
    assert not kq.device_error()
