"""ctypes binding of libkq.so (include/kq.h).  Argument marshalling only.

Loading fails loudly: if the library has not been built (see build.py) a
RuntimeError says so; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

STATUS = {
    0: "KQ_OK", 1: "KQ_ERR_FORMAT", 2: "KQ_ERR_SHAPE", 3: "KQ_ERR_NTOK",
    4: "KQ_ERR_NULL", 5: "KQ_ERR_ALIGN", 6: "KQ_ERR_ALIAS",
    7: "KQ_ERR_CUDA", 8: "KQ_ERR_TIMEOUT", 9: "KQ_ERR_COUNT",
    10: "KQ_ERR_LIMIT", 11: "KQ_ERR_MEMORY",
}
SYMBOLS = ("kq_block_bytes", "kq_matrix_bytes", "kq_matvec",
           "kq_matvec_set", "kq_workspace_bytes", "kq_matvec_set_ws",
           "kq_status_str", "kq_last_cuda_error",
           "kq_device_error", "kq_select_kernel", "kq_set_overlap",
           "kq_last_kernels", "kq_last_launch_count", "kq_matvec_noalloc", "kq_dequant_rows",
           "kq_version")


class KqMat(ctypes.Structure):
    """Mirror of `kq_mat` in include/kq.h."""
    _fields_ = [
        ("fmt", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("W", ctypes.c_void_p),
        ("rows", ctypes.c_int64),
        ("cols", ctypes.c_int64),
        ("x", ctypes.c_void_p),
        ("y", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libkq.so once; raise RuntimeError if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or lib_path()
        if not os.path.exists(p):
            raise RuntimeError(
                f"libkq.so not found at {p}: build it with "
                "`python -m quant_quantized_matvec_gb300.build` (nvcc, "
                "sm_103a); there is no fallback implementation")
        lib = ctypes.CDLL(p)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.kq_block_bytes.argtypes = [i32]
        lib.kq_block_bytes.restype = i64
        lib.kq_matrix_bytes.argtypes = [i32, i64, i64]
        lib.kq_matrix_bytes.restype = i64
        lib.kq_matvec.argtypes = [i32, vp, i64, i64, vp, vp, i32, vp]
        lib.kq_matvec.restype = i32
        lib.kq_dequant_rows.argtypes = [i32, vp, i64, i64, vp, i64, vp, vp]
        lib.kq_dequant_rows.restype = i32
        lib.kq_matvec_noalloc.argtypes = [i32, vp, i64, i64, vp, vp, i32, vp]
        lib.kq_matvec_noalloc.restype = i32
        lib.kq_matvec_set.argtypes = [ctypes.POINTER(KqMat), i32, i32, vp]
        lib.kq_matvec_set.restype = i32
        lib.kq_workspace_bytes.argtypes = [ctypes.POINTER(KqMat), i32, i32]
        lib.kq_workspace_bytes.restype = i64
        lib.kq_matvec_set_ws.argtypes = [ctypes.POINTER(KqMat), i32, i32, vp, vp, i64]
        lib.kq_matvec_set_ws.restype = i32
        lib.kq_status_str.argtypes = [i32]
        lib.kq_status_str.restype = ctypes.c_char_p
        lib.kq_last_cuda_error.argtypes = []
        lib.kq_last_cuda_error.restype = i32
        lib.kq_device_error.argtypes = [i32]
        lib.kq_device_error.restype = i32
        lib.kq_select_kernel.argtypes = [i32]
        lib.kq_select_kernel.restype = i32
        lib.kq_set_overlap.argtypes = [i32]
        lib.kq_set_overlap.restype = i32
        lib.kq_plan_describe.argtypes = [vp, i32, i32, i32, i32, vp, i32]
        lib.kq_plan_describe.restype = i32
        lib.kq_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.kq_set_wait_limit_ns.restype = ctypes.c_ulonglong
        lib.kq_last_kernels.argtypes = []
        lib.kq_last_kernels.restype = i32
        lib.kq_last_launch_count.argtypes = []
        lib.kq_last_launch_count.restype = i32
        lib.kq_version.argtypes = []
        lib.kq_version.restype = i32
        if path is None:
            _lib = lib
        return lib
