"""Inputs with outliers and extreme scales, through the C ABI.

The kernels write each group of 32 inputs in 24-bit fixed point with one
power-of-two step set by the group's largest magnitude, so an outlier
coarsens its group's other inputs.  That rounding adds at most
B = sum_g 2^(E_g - 24) * sum_{j in g} |W_ij| to an output's error (see
envelope.py).  The contract tolerance 1e-4 * sum_j |W_ij x_j| + 1e-6
contains B when the outlier's own product is part of that sum with a weight
that is not tiny -- which random positions give almost always -- but not
when the outlier sits on a zero weight.  Cases:
  * one input per group of 32 scaled by 1e3 at random positions (activation
    outliers): within the contract;
  * whole token columns scaled by 1e30 and by 1e-30 (the step's exponent
    is clamped to [-100, 128]; the tiny column is covered by the absolute
    term): within the contract;
  * one input of 1e4 on a zero weight in every row: within the contract;
  * one input of 1e6 on a zero weight in every row: outside the contract,
    as include/kq.h states, but within the contract widened by B.
Both kernels (streaming and direct) are checked against the oracle.
"""
import numpy as np
import pytest

import gpu_cases as C
from envelope import emulate, zero_weight_at_first_input

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402

FMTS = [kq.Q4_K, kq.Q5_K, kq.Q6_K]
NAMES = {12: "Q4_K", 13: "Q5_K", 14: "Q6_K"}


def run(fmt, W, rows, cols, x, kernel):
    out = C.Guarded(x.shape[0], rows)
    prev = kq.select_kernel(kernel)
    try:
        kq.matvec(fmt, C.to_dev(W), rows, cols, C.to_dev(x), y=out.y)
        torch.cuda.synchronize()
    finally:
        kq.select_kernel(prev)
    assert kq.device_error(clear=True) == 0
    return out.host()


@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_one_outlier_per_group(fmt, kernel):
    rows, cols, ntok = 300, 2816, 2
    W, x = C.case(fmt, rows, cols, ntok, f"outlier/{fmt}")
    x = x.copy()
    rng = np.random.default_rng(fmt)
    groups = x.reshape(ntok, cols // 32, 32)
    pos = rng.integers(0, 32, size=groups.shape[:2])
    for t in range(ntok):
        groups[t, np.arange(groups.shape[1]), pos[t]] *= np.float32(1e3)
    y = run(fmt, W, rows, cols, x, kernel)
    C.check(fmt, W, rows, cols, x, y, what=f"{NAMES[fmt]} {kernel} outliers")


@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_extreme_scales(fmt, kernel):
    rows, cols, ntok = 77, 1280, 2
    W, x = C.case(fmt, rows, cols, ntok, f"scales/{fmt}")
    x = x.copy()
    x[0] *= np.float32(1e30)
    x[1] *= np.float32(1e-30)
    y = run(fmt, W, rows, cols, x, kernel)
    C.check(fmt, W, rows, cols, x, y, what=f"{NAMES[fmt]} {kernel} scales")


@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_outlier_on_a_zero_weight(fmt, kernel):
    rows, cols = 40, 2048
    W = zero_weight_at_first_input(
        fmt, C.case(fmt, rows, cols, 1, f"zw/{fmt}")[0].copy())
    x = C.case(fmt, rows, cols, 1, f"zw/{fmt}")[1].copy()
    x[0, 0] = np.float32(1e4)
    y = run(fmt, W, rows, cols, x, kernel)
    C.check(fmt, W, rows, cols, x, y, what=f"{NAMES[fmt]} {kernel} 1e4 on a zero weight")
    # beyond the envelope: the error is bounded by the rounding bound B
    x[0, 0] = np.float32(1e6)
    y = run(fmt, W, rows, cols, x, kernel)
    err_em, B, tol = emulate(fmt, W, rows, cols, x)
    import oracle
    y_ref, _ = oracle.matvec(fmt, W, rows, cols, x)
    err = np.abs(y.astype(np.float64) - y_ref)
    assert np.all(err <= B + tol), (err / (B + tol)).max()
    assert np.any(err_em > tol)  # the case really is outside the contract
