"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Small cases span several CTAs and ragged tails (row counts that are not a
multiple of the rows a CTA takes, odd block counts per row that leave Q6_K
rows 2-byte aligned); the full-size workloads are the ones the benchmark
times: Q4_K 256x6656; Q4_K/Q5_K/Q6_K 4096x6656 at ntok 1, 2, 4, 8 (every
output); the 202048x6656 Q6_K LM head at ntok 1 and 4 (sampled rows).
The streaming kernel is also compared bitwise with the direct-load kernel,
on small shapes and on the tall Q6_K shapes of its 15-warp launch.
"""
import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402

FMTS = [kq.Q4_K, kq.Q5_K, kq.Q6_K]
NAMES = {12: "Q4_K", 13: "Q5_K", 14: "Q6_K"}


def run(fmt, rows, cols, ntok, label, row_idx=None):
    W, x = C.case(fmt, rows, cols, ntok, label)
    out = C.Guarded(ntok, rows)
    kq.matvec(fmt, C.to_dev(W), rows, cols, C.to_dev(x), y=out.y)
    torch.cuda.synchronize()
    y = out.host()
    C.check(fmt, W, rows, cols, x, y, row_idx=row_idx,
            what=f"{NAMES[fmt]} {rows}x{cols} ntok={ntok}")
    return W, x, y


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
@pytest.mark.parametrize("ntok", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("rows,cols", [(1, 256), (77, 2816), (300, 768),
                                       (33, 9472)])
def test_small_ragged(fmt, ntok, rows, cols):
    run(fmt, rows, cols, ntok, f"small/{fmt}/{rows}/{cols}/{ntok}")


def test_q4k_256x6656():
    run(kq.Q4_K, 256, 6656, 1, "cfg0")


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
@pytest.mark.parametrize("ntok", [1, 2, 4, 8])
def test_4096x6656(fmt, ntok):
    run(fmt, 4096, 6656, ntok, f"cfg2/{fmt}/{ntok}")


@pytest.mark.parametrize("ntok", [1, 4])
def test_lm_head_q6k_sampled(ntok):
    rows, cols = 202048, 6656
    rng = np.random.default_rng(ntok)
    idx = np.unique(np.concatenate([
        [0, 1, 2, 31, 32, 33, rows - 2, rows - 1],
        rng.integers(0, rows, 400)]))
    run(kq.Q6_K, rows, cols, ntok, f"cfg4/{ntok}", row_idx=idx)


def test_overwrites_and_is_deterministic():
    fmt, rows, cols, ntok = kq.Q5_K, 129, 1280, 3
    W, x = C.case(fmt, rows, cols, ntok, "determinism")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    a = C.Guarded(ntok, rows, fill=123.0)
    b = C.Guarded(ntok, rows, fill=float("nan"))
    kq.matvec(fmt, Wd, rows, cols, xd, y=a.y)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kq.matvec(fmt, Wd, rows, cols, xd, y=b.y, stream=s)
    torch.cuda.synchronize()
    ya, yb = a.host(), b.host()
    assert np.array_equal(ya.view(np.uint32), yb.view(np.uint32))
    C.check(fmt, W, rows, cols, x, ya, what="determinism")


def test_rejects_without_launch():
    fmt, rows, cols = kq.Q4_K, 64, 512
    W, x = C.case(fmt, rows, cols, 1, "reject")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    with pytest.raises(kq.KQError, match="KQ_ERR_ALIAS"):
        kq.matvec(fmt, Wd, rows, cols, xd, y=xd.view(-1)[:rows].view(1, rows))
    with pytest.raises(kq.KQError, match="KQ_ERR_NTOK"):
        kq.matvec(fmt, Wd, rows, cols, C.to_dev(np.zeros((17, cols),
                                                          np.float32)))


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
@pytest.mark.parametrize("ntok", [1, 2, 5, 8])
@pytest.mark.parametrize("rows,cols", [(1, 256), (77, 2816), (300, 768),
                                       (33, 9472), (4096, 6656)])
def test_stream_equals_direct(fmt, ntok, rows, cols):
    """The TMA-streaming kernel and the direct-load kernel compute each
    output with the same arithmetic in the same order: bitwise equal."""
    W, x = C.case(fmt, rows, cols, ntok, f"kern/{fmt}/{rows}/{cols}/{ntok}")
    Wd, xd = C.to_dev(W), C.to_dev(x)
    outs = {}
    try:
        for k in ("direct", "stream"):
            kq.select_kernel(k)
            g = C.Guarded(ntok, rows)
            kq.matvec(fmt, Wd, rows, cols, xd, y=g.y)
            torch.cuda.synchronize()
            outs[k] = g.host()
    finally:
        kq.select_kernel("auto")
    assert not kq.device_error()
    assert np.array_equal(outs["direct"].view(np.uint32),
                          outs["stream"].view(np.uint32))
    C.check(fmt, W, rows, cols, x, outs["stream"], what="stream kernel")


@pytest.mark.parametrize("rows,cols,rpt", [(15200, 2560, 1), (6656, 19968, 1),
                                           (39520, 6656, 2)])
def test_tall_q6k_stream_equals_direct(rows, cols, rpt):
    """The 15-warp launch of tall Q6_K sets at one token column, with one
    row a lane-task (row-segment stages: a 15200x2560 matrix, FFN down) and
    with two (whole-row stages: a 39520-row slice of the LM head), against
    the direct-load kernel: bitwise equal, and every output within the
    contract of the oracle."""
    import ctypes
    from quant_quantized_matvec_gb300 import _binding
    fmt, ntok = kq.Q6_K, 1
    lib = _binding.load()
    arr = (_binding.KqMat * 1)()
    arr[0].fmt, arr[0].rows, arr[0].cols = fmt, rows, cols
    arr[0].W = arr[0].x = arr[0].y = 16 << 20  # never read
    out = (ctypes.c_int64 * 64)()
    props = torch.cuda.get_device_properties(0)
    smem = getattr(props, "shared_memory_per_block_optin", 232448)  # GB300: 227 KB
    assert lib.kq_plan_describe(arr, 1, ntok, props.multi_processor_count, smem, out, 64) == 0
    assert out[0] == 0 and out[13] == 15 and out[14] == rpt
    test_stream_equals_direct(fmt, ntok, rows, cols)


@pytest.mark.gpu
def test_overlap_chain_equals_serial():
    """With launch overlap on, each call streams its weights while the call
    before it is still running but reads x only after that call completes.
    A chain whose every input is the previous call's output must give the
    same bits as with overlap off."""
    cols = 1024
    chain = [(kq.Q4_K, "c0"), (kq.Q6_K, "c1"), (kq.Q5_K, "c2"), (kq.Q4_K, "c3")]
    Ws = [C.to_dev(C.case(f, cols, cols, 1, f"chain/{tag}")[0]) for f, tag in chain]
    x0 = C.to_dev(C.case(kq.Q4_K, cols, cols, 1, "chain/x")[1])

    def run():
        ys = [torch.empty((1, cols), dtype=torch.float32, device="cuda") for _ in chain]
        for rep in range(5):
            x = x0
            for (f, _), Wd, y in zip(chain, Ws, ys):
                kq.matvec(f, Wd, cols, cols, x, y=y)
                x = y
        torch.cuda.synchronize()
        return [y.cpu().numpy() for y in ys]

    prev = kq.set_overlap(False)
    try:
        serial = run()
        kq.set_overlap(True)
        overlapped = run()
    finally:
        kq.set_overlap(prev)
    assert not kq.device_error()
    for a, b in zip(serial, overlapped):
        assert np.isfinite(a).all()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
