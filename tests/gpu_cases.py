"""Helpers for the GPU parity tests: seeded inputs on host and device, the
oracle comparison at the contract tolerance, and guarded output buffers."""
from __future__ import annotations

import numpy as np

import oracle
from quant_quantized_matvec_gb300 import synth

# Per-output contract: |y_gpu - y_ref| <= 1e-4 * sum_j |W_ij x_j| + 1e-6.
REL_TOL, ABS_TOL = 1e-4, 1e-6
GUARD = 64  # canary floats on each side of every output


def case(fmt, rows, cols, ntok, label):
    W = synth.kquant_matrix(fmt, rows, cols, f"{label}/W")
    x = synth.activations(ntok, cols, f"{label}/x")
    return W, x


def to_dev(arr):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr).reshape(-1)
                            if arr.dtype == np.uint8 else
                            np.ascontiguousarray(arr)).cuda()


class Guarded:
    """An f32 [ntok, rows] output with NaN canaries around it."""

    def __init__(self, ntok, rows, fill=float("nan")):
        import torch
        self.ntok, self.rows = ntok, rows
        self.buf = torch.full((ntok * rows + 2 * GUARD,), fill,
                              dtype=torch.float32, device="cuda")
        self.buf[:GUARD] = -7.0
        self.buf[-GUARD:] = -7.0
        self.y = self.buf[GUARD:GUARD + ntok * rows].view(ntok, rows)

    def host(self):
        b = self.buf.cpu().numpy()
        assert np.all(b[:GUARD] == -7.0) and np.all(b[-GUARD:] == -7.0), \
            "write outside the output buffer"
        return b[GUARD:GUARD + self.ntok * self.rows].reshape(
            self.ntok, self.rows)


def check(fmt, W, rows, cols, x, y_gpu, row_idx=None, what=""):
    """Compare GPU output rows (all, or row_idx) with the oracle."""
    y_ref, S = oracle.matvec(fmt, W, rows, cols, x, row_idx=row_idx)
    got = y_gpu if row_idx is None else y_gpu[:, row_idx]
    got = got.astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - y_ref)
    tol = REL_TOL * S + ABS_TOL
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (
        f"{what}: {len(bad)} outputs over tolerance, first {bad[:3].tolist()}"
        f" err {err.max():.3e} vs tol {tol.min():.3e}")
    return float((err / np.maximum(S, 1e-30)).max())
