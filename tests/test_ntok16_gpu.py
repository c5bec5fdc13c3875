"""ntok 4..16: the calls that run on the tensor cores, one launch reading W
once for all their token columns.  Parity with the oracle, the independence
of the token columns (bitwise, within each of the two arithmetics), the set
and the no-allocation entry point at these ntok."""
import ctypes

import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402
from quant_quantized_matvec_gb300 import _binding  # noqa: E402

FMTS = (kq.Q4_K, kq.Q5_K, kq.Q6_K)
NAMES = {kq.Q4_K: "q4k", kq.Q5_K: "q5k", kq.Q6_K: "q6k"}


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
@pytest.mark.parametrize("ntok", [9, 12, 16])
@pytest.mark.parametrize("rows,cols", [(1, 256), (77, 2816), (300, 768)])
def test_small_ragged(fmt, ntok, rows, cols):
    W, x = C.case(fmt, rows, cols, ntok, f"n16/{fmt}/{rows}/{cols}/{ntok}")
    g = C.Guarded(ntok, rows)
    kq.matvec(fmt, C.to_dev(W), rows, cols, C.to_dev(x), y=g.y)
    torch.cuda.synchronize()
    C.check(fmt, W, rows, cols, x, g.host(), what=f"{NAMES[fmt]} ntok={ntok}")
    assert not kq.device_error()


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_4096x6656_ntok16(fmt):
    rows, cols, ntok = 4096, 6656, 16
    W, x = C.case(fmt, rows, cols, ntok, f"n16/cfg/{fmt}")
    g = C.Guarded(ntok, rows)
    kq.matvec(fmt, C.to_dev(W), rows, cols, C.to_dev(x), y=g.y)
    torch.cuda.synchronize()
    C.check(fmt, W, rows, cols, x, g.host(), what=f"{NAMES[fmt]} 4096x6656 ntok=16")


@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_token_columns_are_independent(fmt, kernel):
    """A token column's output does not depend on the other columns: column
    t of a 16-column call equals, bit for bit, the same column of a
    5-column call (both on the tensor cores), and column t of a 3-column
    call equals a one-column call (both dp4a), for both kernels."""
    rows, cols, ntok = 193, 3328, 16
    W, x = C.case(fmt, rows, cols, ntok, f"n16/indep/{fmt}")
    Wd = C.to_dev(W)
    try:
        kq.select_kernel(kernel)
        g = C.Guarded(ntok, rows)
        kq.matvec(fmt, Wd, rows, cols, C.to_dev(x), y=g.y)
        quads = []
        for t0 in (0, 5, 11):
            q = C.Guarded(5, rows)
            kq.matvec(fmt, Wd, rows, cols, C.to_dev(x[t0:t0 + 5]), y=q.y)
            quads.append((t0, q))
        g3 = C.Guarded(3, rows)
        kq.matvec(fmt, Wd, rows, cols, C.to_dev(x[2:5]), y=g3.y)
        singles = []
        for t in (2, 4):
            s1 = C.Guarded(1, rows)
            kq.matvec(fmt, Wd, rows, cols, C.to_dev(x[t:t + 1]), y=s1.y)
            singles.append((t, s1))
        torch.cuda.synchronize()
    finally:
        kq.select_kernel("auto")
    y = g.host()
    for t0, q in quads:
        assert np.array_equal(bits(y[t0:t0 + 5]), bits(q.host())), f"columns {t0}.."
    y3 = g3.host()
    for t, s1 in singles:
        assert np.array_equal(bits(y3[t - 2]), bits(s1.host()[0])), f"column {t}"
    C.check(fmt, W, rows, cols, x, y, what=f"{NAMES[fmt]} {kernel} ntok=16")
    assert not kq.device_error()


def test_set_ntok16_equals_separate_calls():
    """A concurrent set at ntok = 16 (Q4_K and Q6_K members sharing x)
    writes what separate calls write."""
    ntok, cols = 16, 2560
    specs = [(kq.Q4_K, 640, "a"), (kq.Q6_K, 96, "b"), (kq.Q5_K, 257, "c")]
    x = C.case(kq.Q4_K, 1, cols, ntok, "n16/set/x")[1]
    xd = C.to_dev(x)
    members, seps, hosts = [], [], []
    for fmt, rows, tag in specs:
        W = C.case(fmt, rows, cols, 1, f"n16/set/{tag}")[0]
        Wd = C.to_dev(W)
        gs, gp = C.Guarded(ntok, rows), C.Guarded(ntok, rows)
        members.append((fmt, Wd, rows, cols, xd, gs.y))
        kq.matvec(fmt, Wd, rows, cols, xd, y=gp.y)
        seps.append((gs, gp))
        hosts.append((fmt, W, rows))
    kq.matvec_set(members)
    torch.cuda.synchronize()
    for (gs, gp), (fmt, W, rows) in zip(seps, hosts):
        ys = gs.host()
        assert np.array_equal(bits(ys), bits(gp.host()))
        C.check(fmt, W, rows, cols, x, ys, what=f"set member {NAMES[fmt]}")
    assert not kq.device_error()


def test_noalloc_ntok12_equals_kq_matvec():
    lib = _binding.load()
    fmt, rows, cols, ntok = kq.Q6_K, 300, 6656, 12
    W, x = C.case(fmt, rows, cols, ntok, "n16/noalloc")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    a, b = C.Guarded(ntok, rows), C.Guarded(ntok, rows)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for fn, g in ((lib.kq_matvec_noalloc, a), (lib.kq_matvec, b)):
        assert fn(fmt, ctypes.c_void_p(Wd.data_ptr()), rows, cols,
                  ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(g.y.data_ptr()),
                  ntok, stream) == 0
    torch.cuda.synchronize()
    assert np.array_equal(bits(a.host()), bits(b.host()))
    C.check(fmt, W, rows, cols, x, a.host(), what="noalloc ntok=12")
    assert not kq.device_error()


@pytest.mark.parametrize("ntok", [2, 3])
@pytest.mark.parametrize("fmt,cols", [(kq.Q6_K, 19968), (kq.Q4_K, 33280)])
def test_wide_matrices_take_the_tensor_cores_from_two_columns(fmt, cols, ntok):
    """At 2 or 3 token columns a matrix whose dp4a input records would not
    stay in shared memory (ntok x cols/256 x record bytes above 140 KB) runs
    on the tensor cores; a narrow one stays on dp4a.  Both match the
    oracle."""
    rows = 200
    W, x = C.case(fmt, rows, cols, ntok, f"wide/{fmt}/{ntok}")
    g = C.Guarded(ntok, rows)
    kq.matvec(fmt, C.to_dev(W), rows, cols, C.to_dev(x), y=g.y)
    torch.cuda.synchronize()
    rec = 1056 if fmt == kq.Q6_K else 832
    assert kq.last_kernels()["tensor_cores"] == (ntok * (cols // 256) * rec > 140 * 1024)
    C.check(fmt, W, rows, cols, x, g.host(), what=f"{NAMES[fmt]} {cols} ntok={ntok}")
    Wn, xn = C.case(fmt, rows, 2560, ntok, f"narrow/{fmt}/{ntok}")
    gn = C.Guarded(ntok, rows)
    kq.matvec(fmt, C.to_dev(Wn), rows, 2560, C.to_dev(xn), y=gn.y)
    torch.cuda.synchronize()
    assert not kq.last_kernels()["tensor_cores"]
    C.check(fmt, Wn, rows, 2560, xn, gn.host(), what=f"{NAMES[fmt]} 2560 ntok={ntok}")
    assert not kq.device_error()


def test_set_mixing_arithmetics_equals_separate_calls():
    """A set at ntok 3 whose wide member runs on the tensor cores and whose
    narrow members run on dp4a: one launch per arithmetic, every output
    bitwise what a separate call writes."""
    ntok = 3
    specs = [(kq.Q4_K, 300, 2560, "a"), (kq.Q6_K, 160, 19968, "b"), (kq.Q5_K, 77, 6656, "c")]
    members, seps, hosts = [], [], []
    for fmt, rows, cols, tag in specs:
        W, x = C.case(fmt, rows, cols, ntok, f"mix/{tag}")
        Wd, xd = C.to_dev(W), C.to_dev(x)
        gs, gp = C.Guarded(ntok, rows), C.Guarded(ntok, rows)
        members.append((fmt, Wd, rows, cols, xd, gs.y))
        kq.matvec(fmt, Wd, rows, cols, xd, y=gp.y)
        seps.append(gp)
        hosts.append((fmt, W, rows, cols, x, gs))
    kq.matvec_set(members, ntok=ntok)
    torch.cuda.synchronize()
    lk = kq.last_kernels()
    assert lk["tensor_cores"] and lk["stream"]
    for (fmt, W, rows, cols, x, gs), gp in zip(hosts, seps):
        assert np.array_equal(bits(gs.host()), bits(gp.host()))
        C.check(fmt, W, rows, cols, x, gs.host(), what="mixed set ntok=3")
    assert not kq.device_error()


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
@pytest.mark.parametrize("rows", [152 * 17, 152 * 27 + 5, 152 * 32, 152 * 45 + 7])
@pytest.mark.parametrize("ntok", [9, 16])
def test_two_tile_units_equal_the_direct_kernel(fmt, rows, ntok):
    """With two octets of tokens the streaming kernel's units span both
    16-row tiles of a group of 17..32 rows and share each fragment load
    (groups of 17, 27-28, 32 and 22-23 rows here, some CTAs one row more):
    every output equals the direct-load kernel's (16-row CTAs, one tile a
    unit) bit for bit, and the oracle's within the tolerance."""
    cols = 2816
    W, x = C.case(fmt, rows, cols, ntok, f"n16/tiles/{fmt}/{rows}/{ntok}")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    outs = {}
    try:
        for kernel in ("stream", "direct"):
            kq.select_kernel(kernel)
            g = C.Guarded(ntok, rows)
            kq.matvec(fmt, Wd, rows, cols, xd, y=g.y)
            torch.cuda.synchronize()
            lk = kq.last_kernels()
            assert lk["tensor_cores"] and lk[kernel]
            outs[kernel] = g.host()
    finally:
        kq.select_kernel("auto")
    assert np.array_equal(bits(outs["stream"]), bits(outs["direct"]))
    C.check(fmt, W, rows, cols, x, outs["stream"], what=f"{NAMES[fmt]} {rows} rows ntok={ntok}")
    assert not kq.device_error()
