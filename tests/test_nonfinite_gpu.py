"""Degenerate inputs through the C ABI: non-finite, zero and subnormal x.

The kernels write x in fixed point with one power-of-two step per group of
32 inputs.  A NaN or infinite input makes its group's step NaN, so every
output of that token column is NaN.  An infinite input has a non-finite
exact result too (the oracle gives an infinity or NaN).  The other token
columns of the same call are untouched and still match the oracle.  An
all-zero column gives exact zeros.  Subnormal inputs sit below the smallest
step: they are read as zero, inside the contract's 1e-6 absolute term.
Both kernels (streaming and direct) and a set sharing x are covered.
"""
import numpy as np
import pytest

import gpu_cases as C
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402

FMTS = [kq.Q4_K, kq.Q5_K, kq.Q6_K]
NAMES = {12: "Q4_K", 13: "Q5_K", 14: "Q6_K"}


def degenerate_x(ntok, cols, label):
    """Token 0: one NaN; 1: one +inf; 2: one -inf; 3: all zero;
    4: subnormal; the rest ordinary N(0,1)."""
    x = C.case(kq.Q4_K, 1, cols, ntok, label)[1].copy()
    x[0, 37] = np.nan
    x[1, cols - 5] = np.inf
    x[2, 300] = -np.inf
    x[3, :] = 0.0
    x[4, :] = np.float32(1e-40) * np.sign(x[4, :])
    return x


def expect(fmt, W, rows, cols, x, y, what):
    y_ref, _ = oracle.matvec(fmt, W, rows, cols, x)
    for t in range(3):
        assert np.isnan(y[t]).all(), f"{what}: token {t} should be all NaN"
        assert not np.isfinite(y_ref[t]).any(), f"{what}: oracle token {t}"
    assert np.array_equal(y[3], np.zeros(rows, np.float32)), f"{what}: zero column"
    C.check(fmt, W, rows, cols, x[4:], y[4:], what=f"{what} (tokens 4..)")


@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_degenerate_inputs(fmt, kernel):
    rows, cols, ntok = 77, 2816, 6
    W = C.case(fmt, rows, cols, ntok, f"degen/{fmt}")[0]
    x = degenerate_x(ntok, cols, f"degen/x/{fmt}")
    out = C.Guarded(ntok, rows, fill=123.0)
    prev = kq.select_kernel(kernel)
    try:
        kq.matvec(fmt, C.to_dev(W), rows, cols, C.to_dev(x), y=out.y)
        torch.cuda.synchronize()
    finally:
        kq.select_kernel(prev)
    expect(fmt, W, rows, cols, x, out.host(), f"{NAMES[fmt]} {kernel}")
    assert kq.device_error(clear=True) == 0


def test_degenerate_inputs_in_a_set():
    cols, ntok = 2816, 5
    x = degenerate_x(ntok, cols, "degen/set/x")
    xd = C.to_dev(x)
    members, host = [], []
    for i, (fmt, rows) in enumerate([(kq.Q4_K, 96), (kq.Q6_K, 40), (kq.Q5_K, 33)]):
        W = C.case(fmt, rows, cols, ntok, f"degen/set/{i}")[0]
        out = C.Guarded(ntok, rows, fill=123.0)
        members.append((fmt, C.to_dev(W), rows, cols, xd, out.y))
        host.append((fmt, W, rows, out))
    kq.matvec_set(members, ntok=ntok)
    torch.cuda.synchronize()
    for fmt, W, rows, out in host:
        expect(fmt, W, rows, cols, x, out.host(), f"set member {NAMES[fmt]}")
    assert kq.device_error(clear=True) == 0
