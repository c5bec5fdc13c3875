"""x and y in pinned host memory: the kernels read and write them in place.
Outputs must be bitwise those of device buffers, for single calls, sets,
both kernels, split calls (ntok > 5) and the no-allocation entry point;
memory the device cannot address is refused before any launch."""
import ctypes

import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402
from quant_quantized_matvec_gb300 import _binding  # noqa: E402

KQ_ERR_MEMORY = 11


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def pinned(shape, fill=np.nan):
    t = torch.full(shape, float(fill), dtype=torch.float32).pin_memory()
    return t


@pytest.mark.parametrize("kernel", ["stream", "direct"])
@pytest.mark.parametrize("fmt,rows,cols,ntok", [(kq.Q4_K, 300, 2816, 1), (kq.Q6_K, 257, 6656, 3),
                                                (kq.Q5_K, 129, 1280, 8)])
def test_host_x_and_y_match_device(fmt, rows, cols, ntok, kernel):
    W, x = C.case(fmt, rows, cols, ntok, f"host/{fmt}/{rows}/{ntok}")
    Wd = C.to_dev(W)
    xh = torch.from_numpy(x).pin_memory()
    try:
        kq.select_kernel(kernel)
        yd = C.Guarded(ntok, rows)
        kq.matvec(fmt, Wd, rows, cols, C.to_dev(x), y=yd.y)
        for xs in (xh, C.to_dev(x)):
            yh = pinned((ntok, rows))
            kq.matvec(fmt, Wd, rows, cols, xs, y=yh)
            torch.cuda.synchronize()
            assert np.array_equal(bits(yh.numpy()), bits(yd.host()))
    finally:
        kq.select_kernel("auto")
    C.check(fmt, W, rows, cols, x, yd.host(), what="device reference")
    assert not kq.device_error()


def test_host_outputs_of_a_set_at_offsets():
    """Set members writing into one pinned buffer at offsets."""
    ntok, cols = 2, 2560
    specs = [(kq.Q4_K, 640), (kq.Q6_K, 96), (kq.Q5_K, 257)]
    x = C.case(kq.Q4_K, 1, cols, ntok, "host/set/x")[1]
    xd = C.to_dev(x)
    total = sum(r for _, r in specs) * ntok
    yh_all = pinned((total + 7,))
    members, refs, off = [], [], 3
    for i, (fmt, rows) in enumerate(specs):
        Wd = C.to_dev(C.case(fmt, rows, cols, 1, f"host/set/W{i}")[0])
        yh = yh_all[off:off + ntok * rows].view(ntok, rows)
        off += ntok * rows
        members.append((fmt, Wd, rows, cols, xd, yh))
        g = C.Guarded(ntok, rows)
        kq.matvec(fmt, Wd, rows, cols, xd, y=g.y)
        refs.append(g)
    kq.matvec_set(members)
    torch.cuda.synchronize()
    for (_, _, _, _, _, yh), g in zip(members, refs):
        assert np.array_equal(bits(yh.numpy()), bits(g.host()))
    assert np.isnan(yh_all[:3].numpy()).all() and np.isnan(yh_all[off:].numpy()).all()
    assert not kq.device_error()


def test_noalloc_with_host_output():
    lib = _binding.load()
    fmt, rows, cols, ntok = kq.Q4_K, 200, 4096, 2
    W, x = C.case(fmt, rows, cols, ntok, "host/noalloc")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    yh = pinned((ntok, rows))
    yd = C.Guarded(ntok, rows)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for fn, y in ((lib.kq_matvec_noalloc, yh.data_ptr()), (lib.kq_matvec, yd.y.data_ptr())):
        assert fn(fmt, ctypes.c_void_p(Wd.data_ptr()), rows, cols, ctypes.c_void_p(xd.data_ptr()),
                  ctypes.c_void_p(y), ntok, s) == 0
    torch.cuda.synchronize()
    assert np.array_equal(bits(yh.numpy()), bits(yd.host()))


def test_noalloc_reads_host_inputs_in_place():
    """kq_matvec_noalloc does not stage host inputs (that would allocate): its
    kernels read x across the host link; the results are the same."""
    lib = _binding.load()
    fmt, rows, cols, ntok = kq.Q6_K, 150, 2560, 3
    W, x = C.case(fmt, rows, cols, ntok, "host/noalloc/x")
    Wd = C.to_dev(W)
    xh = torch.from_numpy(x).pin_memory()
    ya, yb = C.Guarded(ntok, rows), C.Guarded(ntok, rows)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for fn, xp, g in ((lib.kq_matvec_noalloc, xh.data_ptr(), ya),
                      (lib.kq_matvec, C.to_dev(x).data_ptr(), yb)):
        assert fn(fmt, ctypes.c_void_p(Wd.data_ptr()), rows, cols, ctypes.c_void_p(xp),
                  ctypes.c_void_p(g.y.data_ptr()), ntok, s) == 0
    torch.cuda.synchronize()
    assert np.array_equal(bits(ya.host()), bits(yb.host()))


def test_staged_inputs_shared_and_separate_in_a_set():
    """Host inputs of a set, one shared by two members and one of its own,
    each staged once; with overlap on and off."""
    ntok, cols = 3, 1536
    xa = C.case(kq.Q4_K, 1, cols, ntok, "host/stage/xa")[1]
    xb = C.case(kq.Q4_K, 1, cols, ntok, "host/stage/xb")[1]
    xah, xbh = torch.from_numpy(xa).pin_memory(), torch.from_numpy(xb).pin_memory()
    specs = [(kq.Q4_K, 300, xah, xa), (kq.Q6_K, 77, xah, xa), (kq.Q5_K, 129, xbh, xb)]
    prev = kq.set_overlap(False)
    try:
        for overlap in (False, True):
            kq.set_overlap(overlap)
            members, refs = [], []
            for i, (fmt, rows, xh, x) in enumerate(specs):
                Wd = C.to_dev(C.case(fmt, rows, cols, 1, f"host/stage/W{i}")[0])
                g = C.Guarded(ntok, rows)
                members.append((fmt, Wd, rows, cols, xh, g.y))
                ref = C.Guarded(ntok, rows)
                kq.matvec(fmt, Wd, rows, cols, C.to_dev(x), y=ref.y)
                refs.append((g, ref))
            kq.matvec_set(members)
            assert kq.last_launch_count() == 2  # the staging kernel and the set
            torch.cuda.synchronize()
            for g, ref in refs:
                assert np.array_equal(bits(g.host()), bits(ref.host()))
    finally:
        kq.set_overlap(prev)
    assert not kq.device_error()


def test_refuses_memory_the_device_cannot_address():
    """Pageable host memory for y or x, and W outside device memory, return
    KQ_ERR_MEMORY with nothing launched (the output is left untouched)."""
    lib = _binding.load()
    fmt, rows, cols, ntok = kq.Q4_K, 64, 512, 1
    W, x = C.case(fmt, rows, cols, ntok, "host/refuse")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    pageable_y = np.full((ntok, rows), 5.0, dtype=np.float32)
    pageable_x = np.ascontiguousarray(x)
    assert pageable_x.ctypes.data % 16 == 0
    Wh = torch.from_numpy(W.reshape(-1)).pin_memory()
    yd = C.Guarded(ntok, rows, fill=2.0)
    calls = [
        (Wd.data_ptr(), xd.data_ptr(), pageable_y.ctypes.data),
        (Wd.data_ptr(), pageable_x.ctypes.data, yd.y.data_ptr()),
        (Wh.data_ptr(), xd.data_ptr(), yd.y.data_ptr()),
    ]
    for w, xp, yp in calls:
        for fn in (lib.kq_matvec, lib.kq_matvec_noalloc):
            assert fn(fmt, ctypes.c_void_p(w), rows, cols, ctypes.c_void_p(xp), ctypes.c_void_p(yp),
                      ntok, s) == KQ_ERR_MEMORY
    torch.cuda.synchronize()
    assert (pageable_y == 5.0).all()
    assert (yd.host() == 2.0).all()
    assert lib.kq_status_str(KQ_ERR_MEMORY).decode().startswith("a pointer")


def test_dequant_rows_refuses_memory_the_device_cannot_address():
    """kq_dequant_rows checks its pointers like kq_matvec: pageable host ids
    or out, and W outside device memory, return KQ_ERR_MEMORY through the C
    ABI with nothing launched; pinned host ids and out are used in place."""
    lib = _binding.load()
    fmt, rows, cols, n = kq.Q4_K, 64, 512, 3
    W, _ = C.case(fmt, rows, cols, 1, "host/rows")
    Wd = C.to_dev(W)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ids_np = np.array([5, 0, 63], dtype=np.int32)
    ids_d = torch.from_numpy(ids_np).cuda()
    out_d = torch.full((n, cols), 2.0, dtype=torch.float32, device="cuda")
    pageable_out = np.full((n, cols), 5.0, dtype=np.float32)
    assert pageable_out.ctypes.data % 16 == 0
    Wh = torch.from_numpy(W.reshape(-1)).pin_memory()
    calls = [
        (Wd.data_ptr(), ids_np.ctypes.data, out_d.data_ptr()),
        (Wd.data_ptr(), ids_d.data_ptr(), pageable_out.ctypes.data),
        (Wh.data_ptr(), ids_d.data_ptr(), out_d.data_ptr()),
    ]
    for w, ip, op in calls:
        assert lib.kq_dequant_rows(fmt, ctypes.c_void_p(w), rows, cols, ctypes.c_void_p(ip),
                                   n, ctypes.c_void_p(op), s) == KQ_ERR_MEMORY
    torch.cuda.synchronize()
    assert (pageable_out == 5.0).all()
    assert bool((out_d == 2.0).all())
    # pinned host ids and out: gathered in place, bit for bit the oracle's rows
    ids_h = torch.from_numpy(ids_np).pin_memory()
    out_h = torch.empty((n, cols), dtype=torch.float32).pin_memory()
    assert lib.kq_dequant_rows(fmt, ctypes.c_void_p(Wd.data_ptr()), rows, cols,
                               ctypes.c_void_p(ids_h.data_ptr()), n,
                               ctypes.c_void_p(out_h.data_ptr()), s) == 0
    torch.cuda.synchronize()
    import oracle
    ref = oracle.dequant_rows(fmt, W, cols, rows=ids_np.tolist())
    assert np.array_equal(out_h.numpy().view(np.uint32), ref.view(np.uint32))
