"""The further release shapes of "Chapter 6 - The kquant family on the
reference lane", Figure 6.6 (n_in -> n_out = cols -> rows), through the
C ABI against the oracle on sampled rows: the FFN gate/up set, FFN down in
Q4_K and Q6_K, the attention output, the Q5_K LM head, the draft k/v set
and the draft fc.  Each set member is also checked bitwise against the
same matrix launched alone."""
import numpy as np
import pytest

import gpu_cases as C

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402

Q4, Q5, Q6 = kq.Q4_K, kq.Q5_K, kq.Q6_K
SHAPES = {
    "ffn_gate_up_set": [(Q4, 19968, 6656), (Q4, 19968, 6656)],
    "ffn_down_q4k": [(Q4, 6656, 19968)],
    "ffn_down_q6k": [(Q6, 6656, 19968)],
    "attn_output_q4k": [(Q4, 6656, 4096)],
    "lm_head_q5k": [(Q5, 202048, 6656)],
    "draft_kv_set": [(Q4, 1024, 6656), (Q6, 1024, 6656)],
    "draft_fc_q4k": [(Q4, 6656, 33280)],
}


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("ntok", [1, 4])
def test_release_shape(name, ntok):
    members = SHAPES[name]
    cols = members[0][2]
    x = C.case(Q4, 1, cols, ntok, f"release/{name}/{ntok}")[1]
    xd = C.to_dev(x)
    Ws, outs, mem = [], [], []
    for i, (f, rows, c) in enumerate(members):
        W = C.case(f, rows, c, 1, f"release/{name}/{i}")[0]
        Ws.append(W)
        g = C.Guarded(ntok, rows)
        outs.append(g)
        mem.append((f, C.to_dev(W), rows, c, xd, g.y))
    kq.matvec_set(mem, ntok=ntok)
    torch.cuda.synchronize()
    rng = np.random.default_rng(len(name) * 31 + ntok)
    for (f, Wd, rows, c, _, _), W, g in zip(mem, Ws, outs):
        y = g.host()
        idx = np.unique(np.concatenate([[0, rows - 1],
                                        rng.integers(0, rows, size=254)]))
        C.check(f, W, rows, c, x, y, row_idx=idx, what=f"{name} ntok={ntok}")
        if len(mem) > 1:  # a set member equals the matrix launched alone
            alone = C.Guarded(ntok, rows)
            kq.matvec(f, Wd, rows, c, xd, y=alone.y)
            torch.cuda.synchronize()
            assert np.array_equal(alone.host().view(np.uint32), y.view(np.uint32))
    assert not kq.device_error()
