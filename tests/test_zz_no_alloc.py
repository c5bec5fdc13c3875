"""kq_matvec_noalloc through the C ABI.

Some callers cannot allocate device memory during a call: code running under
an allocator or a memory budget that forbids hidden allocations, and loops
that must not take an allocator's locks.  kq_matvec_noalloc serves them with
the direct-load kernel and one fixed device buffer for its input records.
Its results must be bitwise those of kq_matvec with the direct-load kernel
selected, on two calls in a row that reuse the buffer, on calls of the
tensor-core path (ntok = 5 and 12, whose input fragments take the buffer),
and with x in pinned host
memory (read in place, since staging would allocate); each is also checked
against the oracle.  Calls beyond the buffer are refused.

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
DIRECT = 1  # kq_select_kernel: always the direct-load kernel


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(fn, fmt, Wd, rows, cols, xp, y, ntok):
    return fn(fmt, ctypes.c_void_p(Wd.data_ptr()), rows, cols,
              ctypes.c_void_p(xp.data_ptr()), ctypes.c_void_p(y.data_ptr()),
              ntok, _stream())


def _direct_reference(lib, fmt, Wd, rows, cols, xd, ntok):
    """kq_matvec's output with the direct-load kernel selected."""
    prev = lib.kq_select_kernel(DIRECT)
    try:
        ref = C.Guarded(ntok, rows)
        assert _call(lib.kq_matvec, fmt, Wd, rows, cols, xd, ref.y, ntok) == KQ_OK
        torch.cuda.synchronize()
        return ref.host()
    finally:
        lib.kq_select_kernel(prev)


CASES = [(kq.Q6_K, 300, 6656, 2, "noalloc/a"),
         (kq.Q4_K, 517, 2816, 5, "noalloc/b"),
         (kq.Q5_K, 133, 1536, 12, "noalloc/c")]


def test_noalloc_calls_in_a_row_bitwise_equal_direct_kq_matvec():
    lib = _binding.load()
    inputs = []
    for fmt, rows, cols, ntok, label in CASES:
        W, x = C.case(fmt, rows, cols, ntok, label)
        inputs.append((fmt, rows, cols, ntok, W, x, C.to_dev(W), C.to_dev(x)))
    # the no-allocation calls back to back on the one buffer, then again
    for rep in range(2):
        outs = []
        for fmt, rows, cols, ntok, W, x, Wd, xd in inputs:
            g = C.Guarded(ntok, rows)
            assert _call(lib.kq_matvec_noalloc, fmt, Wd, rows, cols, xd, g.y, ntok) == KQ_OK
            # the record (or fragment) pass and the kernel
            assert lib.kq_last_launch_count() == 2
            outs.append(g)
        torch.cuda.synchronize()
        for (fmt, rows, cols, ntok, W, x, Wd, xd), g in zip(inputs, outs):
            y_na = g.host()
            y_mv = _direct_reference(lib, fmt, Wd, rows, cols, xd, ntok)
            assert np.array_equal(y_na.view(np.uint32), y_mv.view(np.uint32)), (rep, fmt)
            C.check(fmt, W, rows, cols, x, y_na, what=f"kq_matvec_noalloc call {rep}")
    assert not kq.device_error()


def test_noalloc_reads_pinned_host_x_in_place():
    lib = _binding.load()
    fmt, rows, cols, ntok = kq.Q4_K, 250, 2560, 3
    W, x = C.case(fmt, rows, cols, ntok, "noalloc/host")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    xh = torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    g = C.Guarded(ntok, rows)
    assert _call(lib.kq_matvec_noalloc, fmt, Wd, rows, cols, xh, g.y, ntok) == KQ_OK
    torch.cuda.synchronize()
    y_na = g.host()
    y_mv = _direct_reference(lib, fmt, Wd, rows, cols, xd, ntok)
    assert np.array_equal(y_na.view(np.uint32), y_mv.view(np.uint32))
    C.check(fmt, W, rows, cols, x, y_na, what="kq_matvec_noalloc, host x")
    assert not kq.device_error()


def test_noalloc_rejects_records_beyond_its_buffer():
    lib = _binding.load()
    ntok, fmt = 8, kq.Q6_K
    # tensor-core records of one octet, 8704 bytes per 256 inputs, above
    # 1 MiB  ->  cols = 256 * 125
    cols = 256 * 125
    assert (cols // 256) * 8704 > NOALLOC_RECORD_BYTES
    rows = 2
    W, x = C.case(fmt, rows, cols, ntok, "noalloc/limit")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    y = torch.full((ntok, rows), 3.0, dtype=torch.float32, device="cuda")
    assert _call(lib.kq_matvec_noalloc, fmt, Wd, rows, cols, xd, y,
                 ntok) == KQ_ERR_LIMIT
    torch.cuda.synchronize()
    assert torch.all(y == 3.0), "a rejected call wrote its output"
    assert lib.kq_status_str(KQ_ERR_LIMIT).decode().startswith("a fixed buffer is too small")
