"""CPU oracle for the K-quant matvec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product (the CUDA library under
``quant_quantized_matvec_gb300/`` and its binding) never imports it, and the
two share no code.

The arithmetic lives in ``kq_oracle.c`` (plain C, gcc, ``-ffp-contract=off``):
block dequantizers that follow "Chapter 6 - The kquant family on the reference
lane" (section 6.2's Q4_K dequantizer, Figures 6.2-6.5) and a matvec that sums
each dot product in f64 in element order ("Chapter 13 - The QKV + gate matvec
family", section 13.1).  This module only compiles that file and marshals
numpy arrays into it.

Parity status: Q4_K is pinned to the worked example of Chapter 6 section 6.3.
Q5_K's high-bit order and Q6_K's code order are readings (R1, R2 in the C
header); their formulas are pinned by closed-form blocks, but agreement with
files written by other software is *parity unpinned*.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kq_oracle.c")
_HDR = os.path.join(_HERE, "kq_oracle.h")
_LIB = os.path.join(_HERE, "_build", "libkq_oracle.so")

Q4_K, Q5_K, Q6_K = 12, 13, 14
FORMATS = (Q4_K, Q5_K, Q6_K)


def compile_library(src: str, out: str, extra_flags=()) -> str:
    """gcc one oracle source file into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-Wall",
           "-shared", "-fPIC", "-I", _HERE, *extra_flags, src, "-o", tmp,
           "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile kq_oracle.c (seconds) unless the library is current."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        compile_library(_SRC, _LIB)
    return _LIB


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """ctypes view of one build of kq_oracle.c."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.kqo_block_bytes.argtypes = [i32]
        lib.kqo_block_bytes.restype = i32
        lib.kqo_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.kqo_f16_to_f32.restype = ctypes.c_float
        lib.kqo_scale_min_k4.argtypes = [vp, i32, vp, vp]
        lib.kqo_scale_min_k4.restype = None
        lib.kqo_dequant_block.argtypes = [i32, vp, vp]
        lib.kqo_dequant_block.restype = i32
        lib.kqo_dequant_row.argtypes = [i32, vp, i64, i64, vp]
        lib.kqo_dequant_row.restype = i32
        lib.kqo_matvec_f32.argtypes = [vp, i64, i64, vp, i32, vp, vp]
        lib.kqo_matvec_f32.restype = None
        lib.kqo_matvec_rows.argtypes = [i32, vp, i64, i64, vp, i32, vp,
                                        i64, vp, vp]
        lib.kqo_matvec_rows.restype = i32
        self.lib = lib

    def block_bytes(self, fmt: int) -> int:
        return int(self.lib.kqo_block_bytes(int(fmt)))

    def f16_to_f32(self, bits: int) -> float:
        return float(self.lib.kqo_f16_to_f32(int(bits) & 0xFFFF))

    def scale_min_k4(self, scales12, j: int) -> tuple[int, int]:
        s = np.ascontiguousarray(np.asarray(scales12, dtype=np.uint8))
        assert s.size == 12
        sc, m = ctypes.c_int(), ctypes.c_int()
        self.lib.kqo_scale_min_k4(_ptr(s), int(j), ctypes.addressof(sc),
                                  ctypes.addressof(m))
        return sc.value, m.value

    def dequant_block(self, fmt: int, block) -> np.ndarray:
        b = np.ascontiguousarray(np.asarray(block, dtype=np.uint8))
        assert b.size == self.block_bytes(fmt)
        out = np.empty(256, dtype=np.float32)
        if self.lib.kqo_dequant_block(int(fmt), _ptr(b), _ptr(out)) != 0:
            raise ValueError("bad format")
        return out

    def dequant_rows(self, fmt: int, W: np.ndarray, cols: int,
                     rows=None) -> np.ndarray:
        """f32 weights of the given rows (all rows when None), [n, cols]."""
        Wb = np.ascontiguousarray(W.reshape(-1).view(np.uint8))
        nrows = Wb.size // (cols // 256 * self.block_bytes(fmt))
        idx = [int(i) for i in (range(nrows) if rows is None else rows)]
        out = np.empty((len(idx), cols), dtype=np.float32)
        for k, i in enumerate(idx):
            if self.lib.kqo_dequant_row(int(fmt), _ptr(Wb), int(cols), i,
                                        _ptr(out[k])) != 0:
                raise ValueError("bad arguments")
        return out

    def matvec_f32(self, W: np.ndarray, x: np.ndarray):
        """Dense f32 W [rows, cols] times x [ntok, cols]; returns (y, S),
        f64 arrays of shape [ntok, rows]."""
        W = np.ascontiguousarray(W, dtype=np.float32)
        x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
        rows, cols = W.shape
        ntok = x.shape[0]
        assert x.shape[1] == cols
        y = np.empty((ntok, rows), dtype=np.float64)
        S = np.empty_like(y)
        self.lib.kqo_matvec_f32(_ptr(W), rows, cols, _ptr(x), ntok, _ptr(y),
                                _ptr(S))
        return y, S

    def matvec(self, fmt: int, W: np.ndarray, rows: int, cols: int,
               x: np.ndarray, row_idx=None):
        """The K-quant matvec.  W holds rows*(cols/256)*block_bytes bytes, x
        is [ntok, cols] f32.  Returns (y, S), f64 [ntok, n], n = rows or the
        length of row_idx when a subset of rows is asked for."""
        Wb = np.ascontiguousarray(W.reshape(-1).view(np.uint8))
        assert Wb.size == rows * (cols // 256) * self.block_bytes(fmt)
        x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
        ntok = x.shape[0]
        assert x.shape[1] == cols
        if row_idx is None:
            n, idx_ptr, idx_arr = rows, None, None
        else:
            idx_arr = np.ascontiguousarray(np.asarray(row_idx,
                                                      dtype=np.int64))
            n, idx_ptr = idx_arr.size, _ptr(idx_arr)
        y = np.empty((ntok, n), dtype=np.float64)
        S = np.empty_like(y)
        rc = self.lib.kqo_matvec_rows(int(fmt), _ptr(Wb), rows, cols,
                                      _ptr(x), ntok, idx_ptr, n, _ptr(y),
                                      _ptr(S))
        if rc != 0:
            raise ValueError("bad arguments")
        return y, S


_lock = threading.Lock()
_default = None


def get() -> Oracle:
    """The oracle built from kq_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def block_bytes(fmt):
    return get().block_bytes(fmt)


def f16_to_f32(bits):
    return get().f16_to_f32(bits)


def scale_min_k4(scales12, j):
    return get().scale_min_k4(scales12, j)


def dequant_block(fmt, block):
    return get().dequant_block(fmt, block)


def dequant_rows(fmt, W, cols, rows=None):
    return get().dequant_rows(fmt, W, cols, rows)


def matvec_f32(W, x):
    return get().matvec_f32(W, x)


def matvec(fmt, W, rows, cols, x, row_idx=None):
    return get().matvec(fmt, W, rows, cols, x, row_idx)
