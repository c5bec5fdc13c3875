"""kq_matvec_set_ws on the GPU (include/kq.h): with a caller's workspace
every output is bitwise what kq_matvec_set writes, on each path that takes
temporaries -- tensor-core fragments, dp4a records in global memory, staged
host inputs, the direct-load kernel -- also when one workspace serves
consecutive calls without a synchronisation between them and inside a
captured CUDA graph; a workspace in host memory or too small is refused
with nothing enqueued."""
import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402

Q4, Q5, Q6 = kq.Q4_K, kq.Q5_K, kq.Q6_K


def bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def build(specs, ntok, tag, host_x=False):
    """Members (fmt, W, rows, cols, x, y) for specs (fmt, rows, cols, plane);
    members with the same plane share x."""
    planes, members = {}, []
    for i, (fmt, rows, cols, pl) in enumerate(specs):
        W = C.case(fmt, rows, cols, 1, f"{tag}/W{i}")[0]
        if pl not in planes:
            x = torch.from_numpy(C.case(fmt, 1, cols, ntok, f"{tag}/x{pl}")[1])
            planes[pl] = x.pin_memory() if host_x else x.cuda()
        y = torch.empty((ntok, rows), dtype=torch.float32, device="cuda")
        members.append((fmt, C.to_dev(W), rows, cols, planes[pl], y))
    return members


def run(members, ntok, workspace=None):
    for m in members:
        m[5].fill_(float("nan"))
    kq.matvec_set(members, ntok=ntok, workspace=workspace)
    torch.cuda.synchronize()
    return [m[5].cpu().numpy().copy() for m in members]


def garbage_workspace(nbytes):
    return torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")


CASES = {
    # name: (specs, ntok, host x, kernel)
    "dp4a_shared_records": ([(Q4, 640, 2560, 0), (Q6, 96, 2560, 0)], 1, False, "auto"),
    "dp4a_global_records": ([(Q4, 300, 73728, 0)], 1, False, "auto"),
    "tensor_cores_ntok8": ([(Q5, 1000, 2816, 0), (Q6, 200, 2816, 0)], 8, False, "auto"),
    "tensor_cores_ntok16": ([(Q4, 2584, 2816, 0)], 16, False, "auto"),
    "mixed_arithmetics": ([(Q4, 300, 2560, 0), (Q6, 160, 19968, 1), (Q5, 77, 6656, 2)], 3,
                          False, "auto"),
    "direct_kernel": ([(Q4, 640, 2560, 0), (Q6, 96, 2560, 0)], 3, False, "direct"),
    "direct_tensor_cores": ([(Q6, 500, 2816, 0)], 12, False, "direct"),
    "host_inputs": ([(Q4, 640, 2560, 0), (Q5, 96, 2560, 1)], 2, True, "auto"),
    "host_inputs_tensor_cores": ([(Q4, 640, 2560, 0)], 8, True, "auto"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_workspace_call_equals_the_allocating_call(name):
    specs, ntok, host_x, kernel = CASES[name]
    members = build(specs, ntok, f"ws/{name}", host_x)
    prev = kq.select_kernel(kernel)
    try:
        ref = run(members, ntok)
        ws = garbage_workspace(kq.workspace_bytes(members, ntok))
        got = run(members, ntok, workspace=ws)
    finally:
        kq.select_kernel(prev)
    for a, b in zip(ref, got):
        assert np.all(np.isfinite(b))
        assert np.array_equal(bits(a), bits(b))
    assert not kq.device_error()


@pytest.mark.parametrize("name", ["tensor_cores_ntok8", "mixed_arithmetics", "host_inputs"])
def test_one_workspace_serves_consecutive_calls(name):
    """Four calls with different inputs share one workspace on one stream,
    with no synchronisation between them: each call's inputs are built only
    after the call before has finished with the workspace."""
    specs, ntok, host_x, _ = CASES[name]
    sets = [build(specs, ntok, f"ws/seq/{name}/{k}", host_x) for k in range(4)]
    refs = [run(m, ntok) for m in sets]
    ws = garbage_workspace(max(kq.workspace_bytes(m, ntok) for m in sets))
    for m in sets:
        for mm in m:
            mm[5].fill_(float("nan"))
    for m in sets:
        kq.matvec_set(m, ntok=ntok, workspace=ws)
    torch.cuda.synchronize()
    for m, ref in zip(sets, refs):
        for mm, a in zip(m, ref):
            assert np.array_equal(bits(a), bits(mm[5].cpu().numpy()))
    assert not kq.device_error()


def test_workspace_calls_in_a_cuda_graph():
    """Three calls on one workspace captured in a graph (kernels only) and
    replayed, with launch overlap on: the outputs equal eager calls'."""
    specs, ntok = CASES["tensor_cores_ntok8"][:2]
    sets = [build(specs, ntok, f"ws/graph/{k}") for k in range(3)]
    refs = [run(m, ntok) for m in sets]
    ws = garbage_workspace(max(kq.workspace_bytes(m, ntok) for m in sets))
    prev = kq.set_overlap(True)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):  # warm-up outside capture
            for m in sets:
                kq.matvec_set(m, ntok=ntok, stream=s, workspace=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for m in sets:
                kq.matvec_set(m, ntok=ntok, stream=s, workspace=ws)
        for m in sets:
            for mm in m:
                mm[5].fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
    finally:
        kq.set_overlap(prev)
    for m, ref in zip(sets, refs):
        for mm, a in zip(m, ref):
            assert np.array_equal(bits(a), bits(mm[5].cpu().numpy()))
    assert not kq.device_error()


def test_bad_workspaces_are_refused():
    specs, ntok = CASES["tensor_cores_ntok8"][:2]
    members = build(specs, ntok, "ws/bad")
    need = kq.workspace_bytes(members, ntok)
    with pytest.raises(kq.KQError) as e:
        kq.matvec_set(members, ntok=ntok, workspace=garbage_workspace(need - 256))
    assert e.value.status == 10  # KQ_ERR_LIMIT
    host = torch.empty(need, dtype=torch.uint8).pin_memory()
    with pytest.raises(kq.KQError) as e:
        kq.matvec_set(members, ntok=ntok, workspace=host)
    assert e.value.status == 11  # KQ_ERR_MEMORY
    torch.cuda.synchronize()
