"""Failure reporting of the streaming kernel, exercised without any fault.

Every wait of the streaming kernel on a shared-memory barrier is bounded by
wall time.  kq_set_wait_limit_ns (a test hook in include/kq_internal.h)
shortens that limit to far below the time the weights take to arrive, so
the waits expire on purpose.  The kernel must then report, not hang: the
call returns, the device error word reads KQ_ERR_TIMEOUT, every output is
either NaN (rows the CTA could not finish) or correct, the copies it had
issued have landed (the next calls on the same SMs compute normally), and a
call made with the default limit matches the oracle again.  Both
arithmetics are covered: one token column (dp4a) and eight (the tensor-core
launch, after its fragment pass).
"""
import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402
from quant_quantized_matvec_gb300 import _binding  # noqa: E402


def _expiring_call(lib, members, ntok, limit_ns):
    prev_kernel = kq.select_kernel("stream")
    prev_limit = lib.kq_set_wait_limit_ns(limit_ns)
    try:
        kq.matvec_set(members, ntok=ntok)
        torch.cuda.synchronize()
    finally:
        lib.kq_set_wait_limit_ns(prev_limit)
        kq.select_kernel(prev_kernel)


def _nan_or_correct(fmt, W, rows, cols, x, y):
    """Every output is NaN or within the contract; returns the NaN count."""
    nan = np.isnan(y)
    if (~nan).any():
        import oracle
        y_ref, S = oracle.matvec(fmt, W, rows, cols, x)
        err = np.abs(y.astype(np.float64) - y_ref)
        ok = err <= C.REL_TOL * S + C.ABS_TOL
        assert np.all(ok | nan), "an output is neither NaN nor correct"
    return int(nan.sum())


@pytest.mark.parametrize("ntok", [1, 8])
@pytest.mark.parametrize("limit_ns", [1, 200])
def test_expired_waits_are_reported_and_the_next_call_is_correct(limit_ns, ntok):
    lib = _binding.load()
    assert not kq.device_error(clear=True)
    cols = 6656
    shapes = [(kq.Q4_K, 4096), (kq.Q6_K, 256), (kq.Q6_K, 256), (kq.Q4_K, 4096)]
    x = C.case(kq.Q4_K, 1, cols, ntok, f"expiry/x/{ntok}")[1]
    xd = C.to_dev(x)
    host, members = [], []
    for i, (fmt, rows) in enumerate(shapes):
        W, _ = C.case(fmt, rows, cols, 1, f"expiry/W{i}")
        g = C.Guarded(ntok, rows)
        host.append((fmt, W, rows, g))
        members.append((fmt, C.to_dev(W), rows, cols, xd, g.y))
    _expiring_call(lib, members, ntok, limit_ns)
    assert kq.device_error(clear=False), "no expired wait was reported"
    assert kq.device_error(clear=True)      # read and clear
    assert not kq.device_error(clear=False)
    nans = sum(_nan_or_correct(fmt, W, rows, cols, x, g.host())
               for fmt, W, rows, g in host)
    assert nans > 0, "waits expired but no output was marked"
    # the same set with the default limit: every output correct, no report
    for (fmt, W, rows, g), m in zip(host, members):
        g.y.fill_(float("nan"))
    kq.matvec_set(members, ntok=ntok)
    torch.cuda.synchronize()
    for fmt, W, rows, g in host:
        C.check(fmt, W, rows, cols, x, g.host(), what="after an expired call")
    assert not kq.device_error()


def test_default_limit_is_restored_and_reported_clear():
    lib = _binding.load()
    assert lib.kq_set_wait_limit_ns(0) == 0   # default in effect
    assert lib.kq_set_wait_limit_ns(0) == 0
    fmt, rows, cols, ntok = kq.Q6_K, 512, 2560, 2
    W, x = C.case(fmt, rows, cols, ntok, "expiry/default")
    y = kq.matvec(fmt, C.to_dev(W), rows, cols, C.to_dev(x))
    torch.cuda.synchronize()
    C.check(fmt, W, rows, cols, x, y.cpu().numpy(), what="default limit")
    assert not kq.device_error()


@pytest.mark.parametrize("rows,cols,rpt", [(15200, 2560, 1), (39520, 6656, 2)])
@pytest.mark.parametrize("limit_ns", [1, 200])
def test_expired_waits_in_the_launch_for_tall_q6k_sets(limit_ns, rows, cols, rpt):
    """The same report from the one-column launch that a Q6_K-only set
    whose CTAs stream 8 or more stages gets (15 consumer warps), with one
    row a lane-task (row-segment stages) and with two (whole-row stages)."""
    import ctypes
    lib = _binding.load()
    fmt, ntok = kq.Q6_K, 1
    arr = (_binding.KqMat * 1)()
    arr[0].fmt, arr[0].rows, arr[0].cols = fmt, rows, cols
    arr[0].W = arr[0].x = arr[0].y = 16 << 20  # never read
    out = (ctypes.c_int64 * 64)()
    props = torch.cuda.get_device_properties(0)
    smem = getattr(props, "shared_memory_per_block_optin", 232448)  # GB300: 227 KB
    assert lib.kq_plan_describe(arr, 1, ntok, props.multi_processor_count, smem, out, 64) == 0
    assert out[0] == 0 and out[13] == 15  # planned, 15 consumer warps
    assert out[14] == rpt                 # rows a lane-task
    assert not kq.device_error(clear=True)
    W, x = C.case(fmt, rows, cols, ntok, "expiry/tall")
    g = C.Guarded(ntok, rows)
    members = [(fmt, C.to_dev(W), rows, cols, C.to_dev(x), g.y)]
    _expiring_call(lib, members, ntok, limit_ns)
    assert kq.device_error(clear=True), "no expired wait was reported"
    assert _nan_or_correct(fmt, W, rows, cols, x, g.host()) > 0
    g.y.fill_(float("nan"))
    kq.matvec_set(members, ntok=ntok)
    torch.cuda.synchronize()
    C.check(fmt, W, rows, cols, x, g.host(), what="tall Q6_K set after an expired call")
    assert not kq.device_error()
