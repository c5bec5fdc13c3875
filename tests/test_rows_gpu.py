"""kq_dequant_rows (the embedding lookup, Chapter 6 section 6.7) against
the oracle's dequantizer, bit for bit: every weight is the correctly
rounded value of d*sc*q - dmin*m (Q4_K, Q5_K) or d*sc*(q-32) (Q6_K), so the
GPU and the oracle must agree exactly (reading R4)."""
import numpy as np
import pytest

import gpu_cases as C
import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import quant_quantized_matvec_gb300 as kq  # noqa: E402

FMTS = [kq.Q4_K, kq.Q5_K, kq.Q6_K]
NAMES = {12: "Q4_K", 13: "Q5_K", 14: "Q6_K"}


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
@pytest.mark.parametrize("rows,cols", [(1, 256), (300, 2816), (77, 6656)])
def test_rows_bitwise_equal_oracle(fmt, rows, cols):
    W, _ = C.case(fmt, rows, cols, 1, f"rows/{fmt}/{rows}/{cols}")
    rng = np.random.default_rng(rows * 7 + cols)
    ids = np.concatenate([[0, rows - 1, rows - 1],
                          rng.integers(0, rows, size=13)]).astype(np.int32)
    out = kq.dequant_rows(fmt, C.to_dev(W), rows, cols,
                          torch.from_numpy(ids).cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = oracle.dequant_rows(fmt, W, cols, rows=ids.tolist())
    assert got.shape == ref.shape
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS, ids=NAMES.get)
def test_rows_out_of_range_ids_give_nan(fmt):
    rows, cols = 5, 512
    W, _ = C.case(fmt, rows, cols, 1, f"rows/nan/{fmt}")
    ids = np.array([2, -1, 5, 4, 1 << 30], dtype=np.int32)
    out = kq.dequant_rows(fmt, C.to_dev(W), rows, cols, torch.from_numpy(ids).cuda())
    got = out.cpu().numpy()
    ref = oracle.dequant_rows(fmt, W, cols, rows=[2, 4])
    assert np.array_equal(got[0].view(np.uint32), ref[0].view(np.uint32))
    assert np.array_equal(got[3].view(np.uint32), ref[1].view(np.uint32))
    assert np.isnan(got[1]).all() and np.isnan(got[2]).all() and np.isnan(got[4]).all()


def test_rows_embedding_table_size():
    """An embedding-table-sized Q4_K matrix (202048 x 6656, 756 MB):
    sampled token rows, bit for bit."""
    rows, cols = 202048, 6656
    W, _ = C.case(kq.Q4_K, rows, cols, 1, "rows/embed")
    ids = np.array([0, 1, 101, 202047, 150000, 77777, 3, 3], dtype=np.int32)
    out = kq.dequant_rows(kq.Q4_K, C.to_dev(W), rows, cols,
                          torch.from_numpy(ids).cuda())
    got = out.cpu().numpy()
    ref = oracle.dequant_rows(kq.Q4_K, W, cols, rows=ids.tolist())
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_rows_rejects():
    fmt, rows, cols = kq.Q4_K, 64, 512
    W, _ = C.case(fmt, rows, cols, 1, "rows/rej")
    Wd = C.to_dev(W)
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(kq.KQError, match="KQ_ERR_ALIAS"):
        kq.dequant_rows(fmt, Wd, rows, cols, ids,
                        out=Wd.view(torch.float32)[:4 * cols].view(4, cols))
    assert kq.dequant_rows(fmt, Wd, rows, cols,
                           torch.zeros(0, dtype=torch.int32, device="cuda")).shape == (0, cols)
