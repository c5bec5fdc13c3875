"""Where the kernels' fixed-point inputs keep the contract, and where not.

The CUDA kernels write each group of 32 consecutive inputs in 24-bit fixed
point with one power-of-two step u = 2^(E-23), 2^(E-1) <= max|x| < 2^E (E
clamped to [-100, 128]), so each input moves by at most u/2 = 2^(E-24).  An
output's error from that rounding is therefore at most

    B = sum_g 2^(E_g - 24) * sum_{j in g} |w_j|

and the contract |y - y_ref| <= 1e-4 * sum_j |w_j x_j| + 1e-6 holds by this
bound whenever B stays below it (plus the much smaller f32 rounding of the
sub-block sums).  A group whose largest input sits on a zero weight adds to
B but not to sum |w x|: that is the case that leaves the contract.

These tests emulate the rounding in numpy (test code: not the oracle, and
not the CUDA path) on top of the oracle's dequantized weights, and pin:
  * for the stated inputs (x ~ N(0,1)), B is hundreds of times inside the
    tolerance, for every format;
  * the emulated error never exceeds B;
  * one input of 1e4 on a zero weight (others N(0,1)) stays inside the
    tolerance; one input of 1e6 on a zero weight breaks it, for every seed.
The precondition in include/kq.h states this envelope.
"""
import numpy as np
import pytest

import oracle
from quant_quantized_matvec_gb300 import synth

from envelope import (BB, FMTS, NAMES, Q6_K, emulate, rounded_inputs,  # noqa: E402,F401
                      zero_weight_at_first_input)


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_stated_inputs_are_far_inside(fmt):
    rows, cols, ntok = 64, 6656, 2
    W = synth.kquant_matrix(fmt, rows, cols, f"envelope/{fmt}")
    x = synth.activations(ntok, cols, f"envelope/x{fmt}")
    err, B, tol = emulate(fmt, W, rows, cols, x)
    assert np.all(err <= B)
    assert np.all(B <= tol / 100), (B / tol).max()


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_zero_weight_outlier_envelope(fmt):
    rows, cols = 8, 1024
    W = zero_weight_at_first_input(
        fmt, synth.kquant_matrix(fmt, rows, cols, f"envelope/zw{fmt}").copy())
    assert np.all(oracle.dequant_rows(fmt, W, cols)[:, 0] == 0.0)
    for seed in range(10):
        x = synth.activations(1, cols, f"envelope/zx{fmt}/{seed}").copy()
        x[0, 0] = np.float32(1e4)
        err, B, tol = emulate(fmt, W, rows, cols, x)
        assert np.all(err <= B)
        assert np.all(err <= tol), f"1e4: {(err / tol).max():.3f} of the tolerance"
        x[0, 0] = np.float32(1e6)
        err, B, tol = emulate(fmt, W, rows, cols, x)
        assert np.all(err <= B)
        assert np.any(err > tol), "1e6 on a zero weight should leave the contract"


def test_rounding_matches_its_definition_on_hand_values():
    """Hand-checked steps: a group whose max is 1.5 has E = 1 (1.5 < 2^1),
    u = 2^-22; a group of zeros takes the smallest step, E = -100."""
    x = np.zeros((1, 64), dtype=np.float32)
    x[0, 0], x[0, 1], x[0, 2] = 1.5, 2.0 ** -22 * 0.49, 2.0 ** -22 * 0.51
    xh, E = rounded_inputs(x)
    assert E.tolist() == [[1, -100]]
    assert xh[0, 0] == 1.5 and xh[0, 1] == 0.0 and xh[0, 2] == 2.0 ** -22
    assert np.all(xh[0, 32:] == 0.0)
    # the largest representable X is 2^23 - 1 steps: max|x| just below 2^E
    x = np.full((1, 32), np.float32(np.nextafter(np.float32(2.0), np.float32(0))))
    xh, E = rounded_inputs(x)
    assert E[0, 0] == 1 and np.all(xh == (2.0 ** 23 - 1) * 2.0 ** -22)
