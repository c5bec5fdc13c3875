"""kq_matvec_set: one launch for several matrices.

  * The QKV+gate concurrent set ("Chapter 13 - The QKV + gate matvec
    family", section 13.5): Q and gate 4096x6656 Q4_K, K and V 256x6656
    Q6_K, one shared x, four outputs.
  * The grid-split pair (audit note "opus_gdn_qsa", section 1): Q6_K and
    Q5_K 2560 -> 512, each with its own x plane, ntok 1..8.
Every member must match the oracle within tolerance and be bitwise equal to
the same matrix run alone.  As in that note's parity check, the test is
shown to catch a pair that reads the wrong input plane: the oracle's answer
for W2 through x1 is far outside tolerance of what the GPU returns.
"""
import numpy as np
import pytest

import gpu_cases as C
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402


def separate(members, ntok):
    outs = []
    for fmt, Wd, rows, cols, xd, _ in members:
        g = C.Guarded(ntok, rows)
        kq.matvec(fmt, Wd, rows, cols, xd, y=g.y)
        outs.append(g)
    torch.cuda.synchronize()
    return [g.host() for g in outs]


def run_set(specs, ntok, label, shared_x=True):
    """specs: list of (fmt, rows, cols).  Returns host data and outputs."""
    host, members, guards = [], [], []
    x_shared = None
    for i, (fmt, rows, cols) in enumerate(specs):
        W, x = C.case(fmt, rows, cols, ntok, f"{label}/{i}")
        if shared_x:
            if x_shared is None:
                x_shared = (x, C.to_dev(x))
            x, xd = x_shared
        else:
            xd = C.to_dev(x)
        g = C.Guarded(ntok, rows)
        members.append((fmt, C.to_dev(W), rows, cols, xd, g.y))
        host.append((fmt, W, rows, cols, x))
        guards.append(g)
    kq.matvec_set(members, ntok=ntok)
    torch.cuda.synchronize()
    return host, members, [g.host() for g in guards]


def test_qkv_gate_set():
    specs = [(kq.Q4_K, 4096, 6656), (kq.Q6_K, 256, 6656),
             (kq.Q6_K, 256, 6656), (kq.Q4_K, 4096, 6656)]
    host, members, outs = run_set(specs, 1, "cfg1")
    alone = separate(members, 1)
    for (fmt, W, rows, cols, x), y, y1 in zip(host, outs, alone):
        assert np.array_equal(y.view(np.uint32), y1.view(np.uint32))
        C.check(fmt, W, rows, cols, x, y, what=f"set member {fmt}x{rows}")


@pytest.mark.parametrize("ntok", [1, 2, 3, 4, 5, 6, 7, 8])
def test_cat_pair_q6k_q5k(ntok):
    specs = [(kq.Q6_K, 512, 2560), (kq.Q5_K, 512, 2560)]
    host, members, outs = run_set(specs, ntok, f"cfg3/{ntok}",
                                  shared_x=False)
    alone = separate(members, ntok)
    for (fmt, W, rows, cols, x), y, y1 in zip(host, outs, alone):
        assert np.array_equal(y.view(np.uint32), y1.view(np.uint32))
        C.check(fmt, W, rows, cols, x, y, what=f"cat {fmt} ntok={ntok}")
    # the comparison would catch W2 read through the first x plane
    fmt2, W2, rows2, cols2, _ = host[1]
    wrong, S = oracle.matvec(fmt2, W2, rows2, cols2, host[0][4])
    err = np.abs(outs[1].astype(np.float64) - wrong)
    assert np.mean(err > C.REL_TOL * S + C.ABS_TOL) > 0.9


def test_max_set_mixed():
    rng = np.random.default_rng(5)
    specs = []
    for i in range(kq.MAX_SET):
        fmt = [kq.Q4_K, kq.Q5_K, kq.Q6_K][i % 3]
        specs.append((fmt, int(rng.integers(1, 200)),
                      256 * int(rng.integers(1, 12))))
    # members with different cols cannot share x: give each its own plane
    host, members, outs = run_set(specs, 3, "maxset", shared_x=False)
    alone = separate(members, 3)
    for (fmt, W, rows, cols, x), y, y1 in zip(host, outs, alone):
        assert np.array_equal(y.view(np.uint32), y1.view(np.uint32))
        C.check(fmt, W, rows, cols, x, y, what=f"maxset {fmt} {rows}x{cols}")


def test_members_sharing_weights():
    fmt, rows, cols = kq.Q6_K, 100, 1024
    W, x = C.case(fmt, rows, cols, 2, "shareW")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    a, b = C.Guarded(2, rows), C.Guarded(2, rows)
    kq.matvec_set([(fmt, Wd, rows, cols, xd, a.y),
                   (fmt, Wd, rows, cols, xd, b.y)], ntok=2)
    torch.cuda.synchronize()
    ya, yb = a.host(), b.host()
    assert np.array_equal(ya.view(np.uint32), yb.view(np.uint32))
    C.check(fmt, W, rows, cols, x, ya, what="shared W")
