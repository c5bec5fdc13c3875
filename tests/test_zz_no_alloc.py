"""kq_matvec_noalloc through the C ABI: two calls in a row on the one fixed
record buffer, each compared with kq_matvec on the same inputs at the
contract tolerance (and with the oracle), plus its size limit.

Collected last on purpose (file name) and self-contained, so it passes both
alone in a fresh process -- where its first call sets the buffer up -- and
after the other tests.
"""
import ctypes

import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402
from quant_quantized_matvec_gb300 import _binding  # noqa: E402

KQ_OK, KQ_ERR_LIMIT = 0, 10
NOALLOC_RECORD_BYTES = 1 << 20


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(fn, fmt, Wd, rows, cols, xd, y, ntok):
    return fn(fmt, ctypes.c_void_p(Wd.data_ptr()), rows, cols,
              ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(y.data_ptr()),
              ntok, _stream())


def test_noalloc_two_calls_match_kq_matvec():
    lib = _binding.load()
    cases = [(kq.Q6_K, 300, 6656, 2, "noalloc/a"),
             (kq.Q4_K, 517, 2816, 5, "noalloc/b")]
    inputs = []
    for fmt, rows, cols, ntok, label in cases:
        W, x = C.case(fmt, rows, cols, ntok, label)
        inputs.append((fmt, rows, cols, ntok, W, x, C.to_dev(W), C.to_dev(x)))
    # two no-allocation calls back to back on the shared buffer
    outs = []
    for fmt, rows, cols, ntok, W, x, Wd, xd in inputs:
        g = C.Guarded(ntok, rows)
        assert _call(lib.kq_matvec_noalloc, fmt, Wd, rows, cols, xd, g.y,
                     ntok) == KQ_OK
        outs.append(g)
    torch.cuda.synchronize()
    for (fmt, rows, cols, ntok, W, x, Wd, xd), g in zip(inputs, outs):
        ref = C.Guarded(ntok, rows)
        assert _call(lib.kq_matvec, fmt, Wd, rows, cols, xd, ref.y,
                     ntok) == KQ_OK
        torch.cuda.synchronize()
        y_na, y_mv = g.host(), ref.host()
        _, S = kq_oracle_S(fmt, W, rows, cols, x)
        assert np.all(np.abs(y_na.astype(np.float64) - y_mv) <=
                      C.REL_TOL * S + C.ABS_TOL)
        C.check(fmt, W, rows, cols, x, y_na, what="kq_matvec_noalloc")
    assert not kq.device_error()


def kq_oracle_S(fmt, W, rows, cols, x):
    import oracle
    return oracle.matvec(fmt, W, rows, cols, x)


def test_noalloc_rejects_records_beyond_its_buffer():
    lib = _binding.load()
    ntok, fmt = 8, kq.Q6_K
    # ntok * (cols / 256) * 1056 > 1 MiB  ->  cols = 256 * 125
    cols = 256 * 125
    assert ntok * (cols // 256) * 1056 > NOALLOC_RECORD_BYTES
    rows = 2
    W, x = C.case(fmt, rows, cols, ntok, "noalloc/limit")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    y = torch.full((ntok, rows), 3.0, dtype=torch.float32, device="cuda")
    assert _call(lib.kq_matvec_noalloc, fmt, Wd, rows, cols, xd, y,
                 ntok) == KQ_ERR_LIMIT
    torch.cuda.synchronize()
    assert torch.all(y == 3.0), "a rejected call wrote its output"
    assert lib.kq_status_str(KQ_ERR_LIMIT).decode().startswith("inputs exceed")
