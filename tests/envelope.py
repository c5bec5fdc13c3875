"""The kernels' fixed-point input rounding, emulated in numpy for the
envelope tests (test code: neither the oracle nor the CUDA path).  See
test_fixed_point_envelope.py for what it pins."""
import numpy as np

import oracle

Q4_K, Q5_K, Q6_K = 12, 13, 14
FMTS = [Q4_K, Q5_K, Q6_K]
NAMES = {12: "Q4_K", 13: "Q5_K", 14: "Q6_K"}
BB = {12: 144, 13: 176, 14: 210}


def rounded_inputs(x):
    """The inputs as the kernels' records hold them: (x_hat, E per group)."""
    ntok, cols = x.shape
    g = np.ascontiguousarray(x, dtype=np.float32).reshape(ntok, cols // 32, 32)
    m = np.abs(g).max(axis=2).astype(np.float32)
    biased = (m.view(np.uint32) >> 23).astype(np.int64)
    E = np.clip(np.maximum(biased, 1) - 126, -100, 128)
    X = np.rint(g.astype(np.float64) * np.exp2(23 - E)[..., None])
    X = np.minimum(X, 2.0 ** 23 - 1)
    return (X * np.exp2(E - 23)[..., None]).reshape(ntok, cols), E


def rounding_bound(Wf, E):
    """B[t, i] = sum_g 2^(E_tg - 24) * sum_{j in g} |W_ij|."""
    rows, cols = Wf.shape
    absw = np.abs(Wf).reshape(rows, cols // 32, 32).sum(axis=2)  # [rows, groups]
    return np.exp2(E - 24.0) @ absw.T                              # [ntok, rows]


def emulate(fmt, W, rows, cols, x):
    """-> (emulated error, bound B, tolerance), each [ntok, rows]."""
    Wf = oracle.dequant_rows(fmt, W, cols).astype(np.float64)
    y_ref, S = oracle.matvec(fmt, W, rows, cols, x)
    xh, E = rounded_inputs(x)
    err = np.abs(xh @ Wf.T - y_ref)
    return err, rounding_bound(Wf, E), 1e-4 * S + 1e-6


def zero_weight_at_first_input(fmt, W):
    """Make every row's first weight exactly zero (in place):
    Q4_K / Q5_K: code 0 and min 0 in sub-block 0 (d*sc*0 - dmin*0);
    Q6_K: code 32 (d*sc*(32 - 32))."""
    for r in range(W.shape[0]):
        b = W[r, 0:BB[fmt]]
        if fmt == Q6_K:
            b[0] &= 0xF0                      # ql[0] low nibble: code bits 0..3
            b[128] = (b[128] & 0xFC) | 2      # qh[0] bits 0..1: code bits 4..5
        else:
            b[8] &= 0xC0                      # scales[4]: m_0 = 0
            qs = 48 if fmt == Q5_K else 16
            b[qs] &= 0xF0                     # qs[0] low nibble: element 0
            if fmt == Q5_K:
                b[16] &= 0xFE                 # qh[0] bit 0: element 0's fifth bit
    return W
