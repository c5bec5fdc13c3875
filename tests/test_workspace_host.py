"""kq_workspace_bytes and kq_matvec_set_ws's argument checks, on the host
with no GPU (include/kq.h): the size is the documented upper bound -- every
member's x as if staged, the tensor-core fragments of the members computed
on the tensor cores, the dp4a records of the largest token chunk -- and a
workspace that is too small, null, misaligned or overlapping a member is
refused before any CUDA call."""
import ctypes

import pytest

from quant_quantized_matvec_gb300 import _binding

Q4, Q5, Q6 = 12, 13, 14
REC = {Q4: 832, Q5: 832, Q6: 1056}   # dp4a record bytes per token and 256 inputs
FRAG = 8704                          # tensor-core bytes per octet of tokens and 256 inputs
LIMIT, NULL, ALIGN, ALIAS, NTOK = 10, 4, 5, 6, 3


def r256(b):
    return -(-b // 256) * 256


def on_tensor_cores(fmt, cols, ntok):
    # the arithmetic choice of kq.h: 4..16 columns, or 2..3 columns whose
    # records would pass 140 KB
    return ntok >= 4 or (ntok >= 2 and ntok * (cols // 256) * REC[fmt] > 140 * 1024)


def expected(members, ntok):
    stage = sum(r256(ntok * cols * 4) for _, _, cols, _ in members)
    planes, tc, dp = set(), 0, 0
    for fmt, rows, cols, x in members:
        nb = cols // 256
        if on_tensor_cores(fmt, cols, ntok):
            if (x, cols) not in planes:
                planes.add((x, cols))
                tc += r256(nb * -(-ntok // 8) * FRAG)
        else:
            dp += r256(min(ntok, 8) * nb * REC[fmt])
    return stage + tc + dp


def descs(members):
    arr = (_binding.KqMat * len(members))()
    base = 1 << 32
    for i, (fmt, rows, cols, x) in enumerate(members):
        arr[i].fmt, arr[i].rows, arr[i].cols = fmt, rows, cols
        arr[i].W = base + (i << 28)              # 16-byte aligned, never read
        arr[i].x = (1 << 40) + (x << 28)          # members may share x
        arr[i].y = (1 << 44) + (i << 28)
    return arr


QKV = [(Q4, 4096, 6656, 0), (Q6, 256, 6656, 0), (Q6, 256, 6656, 0), (Q4, 4096, 6656, 0)]
CASES = [
    (QKV, 1), (QKV, 3), (QKV, 8), (QKV, 16),
    ([(Q6, 160, 19968, 0)], 2),                       # wide: tensor cores at ntok 2
    ([(Q4, 300, 2560, 0), (Q6, 160, 19968, 1), (Q5, 77, 6656, 2)], 3),  # mixed arithmetics
    ([(Q5, 202048, 6656, 0)], 12),
    ([(Q4, 64, 256, 0), (Q4, 64, 256, 1)], 1),
]


@pytest.mark.parametrize("members,ntok", CASES)
def test_workspace_bytes_is_the_documented_bound(members, ntok):
    lib = _binding.load()
    arr = descs(members)
    assert lib.kq_workspace_bytes(arr, len(members), ntok) == expected(members, ntok)


def test_workspace_bytes_rejects_what_the_set_call_rejects():
    lib = _binding.load()
    arr = descs(QKV)
    assert lib.kq_workspace_bytes(arr, 4, 0) == -NTOK
    assert lib.kq_workspace_bytes(arr, 4, 17) == -NTOK
    assert lib.kq_workspace_bytes(arr, 0, 1) == -9   # KQ_ERR_COUNT


def test_set_ws_validates_before_any_cuda_call():
    """These calls return their errors without touching the (absent) GPU."""
    lib = _binding.load()
    arr = descs(QKV)
    need = lib.kq_workspace_bytes(arr, 4, 8)
    ws = 1 << 46
    assert lib.kq_matvec_set_ws(arr, 4, 8, None, ws, need - 1) == LIMIT
    assert lib.kq_matvec_set_ws(arr, 4, 8, None, None, need) == NULL
    assert lib.kq_matvec_set_ws(arr, 4, 8, None, ws + 128, need) == ALIGN
    # over member 0's y
    assert lib.kq_matvec_set_ws(arr, 4, 8, None, arr[0].y - 256, need + 512) == ALIAS
    assert lib.kq_matvec_set_ws(arr, 4, 0, None, ws, need) == NTOK
