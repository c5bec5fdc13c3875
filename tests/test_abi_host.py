"""The C ABI on the host, without a GPU: the library loads, exports every
function include/kq.h declares, and rejects bad arguments before it touches
CUDA (only invalid arguments are passed here, with fake device pointers)."""
import ctypes
import os
import re

import pytest

from quant_quantized_matvec_gb300 import _binding
from quant_quantized_matvec_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, FORMAT, SHAPE, NTOK, NULL, ALIGN, ALIAS, CUDA, TIMEOUT, COUNT, LIMIT, MEMORY = range(12)


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return _binding.load()


def header_functions(name="kq.h"):
    with open(os.path.join(ROOT, "include", name)) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kq_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert set(names) == set(_binding.SYMBOLS)
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            for n in header_functions(h):
                assert hasattr(lib, n), f"{h}: {n}"
    assert header_functions("kq_internal.h") == ["kq_plan_describe", "kq_set_wait_limit_ns"]


def test_block_and_matrix_bytes(lib):
    assert [lib.kq_block_bytes(f) for f in (12, 13, 14)] == [144, 176, 210]
    assert lib.kq_block_bytes(0) == -1 and lib.kq_block_bytes(15) == -1
    assert lib.kq_matrix_bytes(12, 4096, 6656) == 15335424
    assert lib.kq_matrix_bytes(13, 202048, 6656) == 924571648
    assert lib.kq_matrix_bytes(14, 202048, 6656) == 1103182080
    assert lib.kq_matrix_bytes(12, 0, 256) == -1
    assert lib.kq_matrix_bytes(12, 1, 255) == -1
    assert lib.kq_matrix_bytes(12, 1, 1 << 21) == -1
    assert lib.kq_version() >> 16 == 1


def test_status_strings(lib):
    for s in range(12):
        assert lib.kq_status_str(s) != b"unknown status"
    assert lib.kq_status_str(99) == b"unknown status"


def test_status_values_follow_the_boundary(lib):
    """The first nine codes keep the order of the boundary's enum (OK,
    FORMAT, SHAPE, NTOK, NULL, ALIGN, ALIAS, CUDA, TIMEOUT); the library's
    extra codes come after them.  Read from the header text itself."""
    with open(os.path.join(ROOT, "include", "kq.h")) as f:
        src = f.read()
    vals = dict((k, int(v)) for k, v in re.findall(r"\b(KQ_[A-Z_]+) = (\d+)", src))
    assert [vals[k] for k in ("KQ_OK", "KQ_ERR_FORMAT", "KQ_ERR_SHAPE", "KQ_ERR_NTOK",
                              "KQ_ERR_NULL", "KQ_ERR_ALIGN", "KQ_ERR_ALIAS",
                              "KQ_ERR_CUDA", "KQ_ERR_TIMEOUT")] == list(range(9))
    assert (vals["KQ_ERR_COUNT"], vals["KQ_ERR_LIMIT"], vals["KQ_ERR_MEMORY"]) == (9, 10, 11)
    for k, v in vals.items():
        if k.startswith("KQ_ERR_") or k == "KQ_OK":
            assert _binding.STATUS[v] == k
    assert lib.kq_status_str(CUDA).decode().startswith("a CUDA call")
    assert lib.kq_status_str(TIMEOUT).decode().startswith("device-side wait")


# fake, well-aligned device addresses: validation must reject the call
# before any CUDA call, so they are never dereferenced
W0, X0, Y0 = 0x7f0000000000, 0x7f1000000000, 0x7f2000000000


def mv(lib, fmt=12, W=W0, rows=64, cols=512, x=X0, y=Y0, ntok=1):
    return lib.kq_matvec(fmt, W, rows, cols, x, y, ntok, None)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=11), FORMAT), (dict(fmt=0), FORMAT), (dict(fmt=1000), FORMAT),
    (dict(rows=0), SHAPE), (dict(rows=-3), SHAPE), (dict(cols=0), SHAPE),
    (dict(cols=255), SHAPE), (dict(cols=300), SHAPE),
    (dict(cols=1 << 21), SHAPE), (dict(rows=(1 << 30) + 1), SHAPE),
    (dict(ntok=0), NTOK), (dict(ntok=17), NTOK), (dict(ntok=-1), NTOK),
    (dict(W=None), NULL), (dict(x=None), NULL), (dict(y=None), NULL),
    (dict(W=W0 + 8), ALIGN), (dict(x=X0 + 4), ALIGN), (dict(y=Y0 + 2), ALIGN),
    # y overlapping W, or x
    (dict(y=W0 + 64), ALIAS), (dict(y=X0 + 1024), ALIAS),
    (dict(y=X0 - 64), ALIAS),
])
def test_matvec_rejects(lib, kw, status):
    assert mv(lib, **kw) == status


def test_alias_edges(lib):
    # y ending exactly where x begins does not overlap: validation passes and
    # the call would go on to CUDA, so only the failing neighbour is checked
    rows = 64
    assert mv(lib, y=X0 - 4 * rows + 4) == ALIAS
    assert mv(lib, y=W0 + 64 * 2 * 144 - 4) == ALIAS


def _mats(specs):
    arr = (_binding.KqMat * len(specs))()
    for i, s in enumerate(specs):
        d = dict(fmt=12, W=W0 + i * (1 << 28), rows=64, cols=512, x=X0,
                 y=Y0 + i * (1 << 28), reserved=0)
        d.update(s)
        for k, v in d.items():
            setattr(arr[i], k, v)
    return arr


def mvset(lib, specs, ntok=1, n=None):
    arr = _mats(specs)
    return lib.kq_matvec_set(
        ctypes.cast(arr, ctypes.POINTER(_binding.KqMat)),
        len(specs) if n is None else n, ntok, None)


def test_set_rejects(lib):
    assert mvset(lib, [{}], n=0) == COUNT
    assert mvset(lib, [{}] * 17) == COUNT
    assert lib.kq_matvec_set(None, 1, 1, None) == NULL
    assert mvset(lib, [{}, {"fmt": 9}]) == FORMAT
    assert mvset(lib, [{}, {"cols": 100}]) == SHAPE
    assert mvset(lib, [{}, {"reserved": 1}]) == SHAPE
    assert mvset(lib, [{}, {}], ntok=17) == NTOK
    assert mvset(lib, [{}, {"x": None}]) == NULL
    assert mvset(lib, [{}, {"W": W0 + 4}]) == ALIGN
    # two outputs overlapping each other
    assert mvset(lib, [{"y": Y0}, {"y": Y0 + 128}]) == ALIAS
    # one member's output over another member's weights / input plane
    assert mvset(lib, [{}, {"y": W0 + 32}]) == ALIAS
    assert mvset(lib, [{"x": X0}, {"x": X0 + (1 << 20), "y": X0 + 16}]) == ALIAS


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        _binding.load(str(tmp_path / "libkq.so"))


def test_stage_task_division_is_exact():
    """The streaming kernel splits a stage task index t into (block column,
    row pair) as t // hp by multiply-shift: (t * ceil(2^20 / hp)) >> 20 in
    32-bit arithmetic.  The planner keeps t below 2^12 and hp at most 32;
    over that whole range the shortcut must equal the true quotient."""
    for hp in range(1, 33):
        hinv = ((1 << 20) + hp - 1) // hp
        for t in range(4096):
            assert ((t * hinv) & 0xFFFFFFFF) >> 20 == t // hp, (hp, t)


def test_noalloc_validates_before_any_cuda_call():
    """kq_matvec_noalloc checks its arguments and its buffer limit on the
    host: these calls return without touching the (absent) GPU."""
    lib = _binding.load()
    fake = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced
    assert lib.kq_matvec_noalloc(99, fake, 4, 256, fake, ctypes.c_void_p(1 << 24), 1,
                                 None) == 1  # KQ_ERR_FORMAT
    assert lib.kq_matvec_noalloc(14, fake, 4, 255, fake, ctypes.c_void_p(1 << 24), 1,
                                 None) == 2  # KQ_ERR_SHAPE
    # Q6_K records for ntok=8, cols=256*125: 8*125*1056 > 1 MiB
    assert lib.kq_matvec_noalloc(14, ctypes.c_void_p(1 << 30), 2, 256 * 125,
                                 ctypes.c_void_p(1 << 34), ctypes.c_void_p(1 << 36), 8,
                                 None) == 10  # KQ_ERR_LIMIT
    assert lib.kq_status_str(10).decode().startswith("a fixed buffer is too small")


def test_dequant_rows_validates_before_any_cuda_call():
    lib = _binding.load()
    W, ids, out = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 24), ctypes.c_void_p(1 << 28)
    assert lib.kq_dequant_rows(99, W, 4, 256, ids, 1, out, None) == 1   # format
    assert lib.kq_dequant_rows(12, W, 4, 300, ids, 1, out, None) == 2   # cols % 256
    assert lib.kq_dequant_rows(12, W, 4, 256, ids, -1, out, None) == 2  # n < 0
    assert lib.kq_dequant_rows(12, W, 4, 256, None, 0, None, None) == 0  # n = 0: nothing to do
    assert lib.kq_dequant_rows(12, W, 4, 256, None, 1, out, None) == 4  # null ids
    assert lib.kq_dequant_rows(12, W, 4, 256, ids, 1, ctypes.c_void_p((1 << 28) + 4), None) == 5
    assert lib.kq_dequant_rows(12, W, 4, 256, ids, 1, ctypes.c_void_p((1 << 20) + 16), None) == 6
