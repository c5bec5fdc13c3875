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
Calls of 4 or more token columns run on the tensor cores instead, where
each input keeps about 22 significant bits and the rounding floor is
2^(E - 39) for a 256-input column whose largest magnitude is below 2^E
(kq_xtc.cuh): there every case above, the 1e6 outlier included, is within
the contract, and a row whose weights are all exactly zero gives exactly
zero on both paths.
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


@pytest.mark.parametrize("ntok", [2, 8])
@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_one_outlier_per_group(fmt, kernel, ntok):
    rows, cols = 300, 2816
    W, x = C.case(fmt, rows, cols, ntok, f"outlier/{fmt}")
    x = x.copy()
    rng = np.random.default_rng(fmt)
    groups = x.reshape(ntok, cols // 32, 32)
    pos = rng.integers(0, 32, size=groups.shape[:2])
    for t in range(ntok):
        groups[t, np.arange(groups.shape[1]), pos[t]] *= np.float32(1e3)
    y = run(fmt, W, rows, cols, x, kernel)
    C.check(fmt, W, rows, cols, x, y, what=f"{NAMES[fmt]} {kernel} ntok={ntok} outliers")


@pytest.mark.parametrize("ntok", [2, 8])
@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_extreme_scales(fmt, kernel, ntok):
    rows, cols = 77, 1280
    W, x = C.case(fmt, rows, cols, ntok, f"scales/{fmt}")
    x = x.copy()
    x[0] *= np.float32(1e30)
    x[1] *= np.float32(1e-30)
    y = run(fmt, W, rows, cols, x, kernel)
    C.check(fmt, W, rows, cols, x, y, what=f"{NAMES[fmt]} {kernel} ntok={ntok} scales")


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


@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_outlier_on_a_zero_weight_tensor_cores(fmt, kernel):
    """At ntok = 5 (tensor cores) an input of 1e4 and one of 1e6 on a zero
    weight both stay within the contract itself."""
    rows, cols, ntok = 40, 2048, 5
    W = zero_weight_at_first_input(
        fmt, C.case(fmt, rows, cols, 1, f"zw/{fmt}")[0].copy())
    x = C.case(fmt, rows, cols, ntok, f"zw5/{fmt}")[1].copy()
    for big in (1e4, 1e6):
        x[:, 0] = np.float32(big)
        y = run(fmt, W, rows, cols, x, kernel)
        C.check(fmt, W, rows, cols, x, y,
                what=f"{NAMES[fmt]} {kernel} ntok={ntok} {big:g} on a zero weight")


def zero_rows(fmt, W, idx):
    """Make every weight of rows `idx` exactly zero (in place), scales left
    random: Q4_K / Q5_K: all codes 0 and all mins 0 (d*sc*0 - dmin*0);
    Q6_K: all codes 32 (d*sc*(32 - 32))."""
    bb = C.synth.BLOCK_BYTES[fmt]
    blocks = W.reshape(W.shape[0], -1, bb)
    assert np.shares_memory(blocks, W)
    if fmt == kq.Q6_K:
        blocks[idx, :, 0:128] = 0          # ql: code bits 0..3
        blocks[idx, :, 128:192] = 0xAA     # qh: code bits 4..5 = 0b10
    else:
        blocks[idx, :, 8:12] = 0           # scales[4..7]: m_0..3, top bits of m_4..7
        blocks[idx, :, 12:16] &= 0x0F      # scales[8..11]: low bits of m_4..7
        qs = 48 if fmt == kq.Q5_K else 16
        blocks[idx, :, qs:qs + 128] = 0    # code low bits
        if fmt == kq.Q5_K:
            blocks[idx, :, 16:48] = 0      # qh: code bit 4
    return W


@pytest.mark.parametrize("ntok", [1, 3, 8])
@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_zero_weight_rows_give_zero(fmt, kernel, ntok):
    """Rows whose weights are all exactly zero give exactly zero (S = 0, so
    the contract allows only the absolute 1e-6), on the dp4a and the
    tensor-core arithmetic, with ordinary rows around them."""
    rows, cols = 96, 2560
    W, x = C.case(fmt, rows, cols, ntok, f"zrow/{fmt}/{ntok}")
    W = np.ascontiguousarray(W).copy()
    zero_rows(fmt, W, np.arange(0, rows, 3))
    y = run(fmt, W, rows, cols, x, kernel)
    assert np.all(y[:, ::3] == 0.0), np.abs(y[:, ::3]).max()
    C.check(fmt, W, rows, cols, x, y, what=f"{NAMES[fmt]} {kernel} ntok={ntok} zero rows")
