"""GB300 (sm_103a) K-quant matvec: y = W x with W in Q4_K / Q5_K / Q6_K.

Thin Python layer over the C ABI of libkq.so (include/kq.h).  PyTorch
supplies device memory and streams; every step of the computation runs in
the library's CUDA kernels.  The functions take torch CUDA tensors, check
their dtype/shape/device, and pass raw pointers through.

    import quant_quantized_matvec_gb300 as kq
    y = kq.matvec(kq.Q4_K, W, rows, cols, x)          # x: [ntok, cols] f32
    kq.matvec_set([(kq.Q4_K, Wq, 4096, 6656, x, yq), ...])
"""
from __future__ import annotations

import ctypes

from . import _binding

Q4_K, Q5_K, Q6_K = 12, 13, 14
FORMATS = (Q4_K, Q5_K, Q6_K)
MAX_NTOK = 16
MAX_SET = 16
# status codes of include/kq.h that the wrappers act on
KQ_ERR_CUDA, KQ_ERR_TIMEOUT = 7, 8


class KQError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _binding.load()
        msg = lib.kq_status_str(status).decode()
        extra = ""
        if status == KQ_ERR_CUDA:
            extra = f" (cudaError {lib.kq_last_cuda_error()})"
        super().__init__(f"{where}: {_binding.STATUS.get(status, status)}: "
                         f"{msg}{extra}")
        self.status = status


def _lib():
    return _binding.load()


def block_bytes(fmt: int) -> int:
    return int(_lib().kq_block_bytes(int(fmt)))


def matrix_bytes(fmt: int, rows: int, cols: int) -> int:
    return int(_lib().kq_matrix_bytes(int(fmt), int(rows), int(cols)))


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_tensor(t, name, dtype=None, host_ok=False):
    """W must be a CUDA tensor; x and y (host_ok) may also be pinned CPU
    tensors, which the kernels read and write in place."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor"
                         + (" or a pinned CPU tensor" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def matvec(fmt, W, rows, cols, x, y=None, stream=None):
    """y[t, i] = sum_j W[i, j] x[t, j] for the K-quant matrix W (uint8
    bytes, rows*(cols/256)*block_bytes of them), x [ntok, cols] or [cols]
    f32.  Returns y [ntok, rows] (or [rows] for 1-D x), f32."""
    import torch
    squeeze = x.dim() == 1
    x2 = x.unsqueeze(0) if squeeze else x
    _check_tensor(W, "W")
    _check_tensor(x2, "x", torch.float32, host_ok=True)
    ntok = x2.shape[0]
    if x2.shape[1] != cols:
        raise ValueError("x must have cols columns")
    if W.numel() * W.element_size() != matrix_bytes(fmt, rows, cols):
        raise ValueError("W size does not match fmt/rows/cols")
    if y is None:
        y = torch.empty((ntok, rows), dtype=torch.float32,
                        device=x.device if x.is_cuda else "cuda")
    _check_tensor(y, "y", torch.float32, host_ok=True)
    if y.numel() != ntok * rows:
        raise ValueError("y must hold ntok*rows floats")
    st = _lib().kq_matvec(int(fmt), W.data_ptr(), int(rows), int(cols),
                          x2.data_ptr(), y.data_ptr(), int(ntok),
                          _stream_ptr(stream))
    if st != 0:
        raise KQError(st, "kq_matvec")
    return y.view(rows) if squeeze and y.dim() == 2 and ntok == 1 else y


def dequant_rows(fmt, W, rows, cols, ids, out=None, stream=None):
    """Rows ids of the K-quant matrix W, dequantized to f32 [len(ids), cols]
    (the embedding lookup).  ids: int32 tensor on the device."""
    import torch
    _check_tensor(W, "W")
    _check_tensor(ids, "ids", torch.int32)
    n = ids.numel()
    if W.numel() * W.element_size() != matrix_bytes(fmt, rows, cols):
        raise ValueError("W size does not match fmt/rows/cols")
    if out is None:
        out = torch.empty((n, cols), dtype=torch.float32, device=W.device)
    _check_tensor(out, "out", torch.float32)
    if out.numel() != n * cols:
        raise ValueError("out must hold len(ids)*cols floats")
    st = _lib().kq_dequant_rows(int(fmt), W.data_ptr(), int(rows), int(cols),
                                ids.data_ptr(), int(n), out.data_ptr(),
                                _stream_ptr(stream))
    if st != 0:
        raise KQError(st, "kq_dequant_rows")
    return out


def make_set(members):
    """members: iterable of (fmt, W, rows, cols, x, y) with torch tensors.
    Returns a ctypes array of kq_mat descriptors (reusable across calls)."""
    members = list(members)
    arr = (_binding.KqMat * len(members))()
    for i, (fmt, W, rows, cols, x, y) in enumerate(members):
        arr[i].fmt = int(fmt)
        arr[i].reserved = 0
        arr[i].W = W.data_ptr()
        arr[i].rows = int(rows)
        arr[i].cols = int(cols)
        arr[i].x = x.data_ptr()
        arr[i].y = y.data_ptr()
    return arr


def workspace_bytes(members, ntok):
    """Bytes of the device workspace matvec_set(..., workspace=) needs for
    these members (fmt, W, rows, cols, x, y) -- or descriptors from
    make_set -- at ntok token columns (kq_workspace_bytes)."""
    desc = members if isinstance(members, ctypes.Array) else make_set(members)
    n = _lib().kq_workspace_bytes(ctypes.cast(desc, ctypes.POINTER(_binding.KqMat)),
                                  len(desc), int(ntok))
    if n < 0:
        raise KQError(int(n), "kq_workspace_bytes")
    return int(n)


def matvec_set(members, ntok=None, stream=None, descriptors=None, workspace=None):
    """Several matvecs in one launch.  members: list of (fmt, W, rows, cols,
    x, y); x [ntok, cols] f32 (members may share x), y [ntok, rows] f32.
    `descriptors` (from make_set) skips rebuilding the descriptor array.
    `workspace`: a CUDA uint8 tensor of at least workspace_bytes(...) bytes,
    256-byte aligned, taken instead of the library's stream-ordered
    temporaries (kq_matvec_set_ws); it must not be used by another call
    that may run at the same time."""
    import torch
    members = list(members)
    if ntok is None:
        x0 = members[0][4]
        ntok = 1 if x0.dim() == 1 else x0.shape[0]
    if descriptors is None:
        for (fmt, W, rows, cols, x, y) in members:
            _check_tensor(W, "W")
            _check_tensor(x, "x", torch.float32, host_ok=True)
            _check_tensor(y, "y", torch.float32, host_ok=True)
            if x.numel() != ntok * cols or y.numel() != ntok * rows:
                raise ValueError("x / y sizes do not match ntok, rows, cols")
            if W.numel() * W.element_size() != matrix_bytes(fmt, rows, cols):
                raise ValueError("W size does not match fmt/rows/cols")
        descriptors = make_set(members)
    dp = ctypes.cast(descriptors, ctypes.POINTER(_binding.KqMat))
    if workspace is None:
        st = _lib().kq_matvec_set(dp, len(members), int(ntok), _stream_ptr(stream))
        if st != 0:
            raise KQError(st, "kq_matvec_set")
    else:
        st = _lib().kq_matvec_set_ws(dp, len(members), int(ntok), _stream_ptr(stream),
                                     workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size())
        if st != 0:
            raise KQError(st, "kq_matvec_set_ws")
    return [m[5] for m in members]



KERNELS = {"auto": 0, "direct": 1, "stream": 2}


def select_kernel(which: str) -> str:
    """Choose the kernel ("auto", "direct", "stream"); returns the previous
    choice.  Results are identical for every choice."""
    prev = _lib().kq_select_kernel(KERNELS[which])
    return {v: k for k, v in KERNELS.items()}[prev]


def last_kernels() -> dict:
    """Kernels enqueued by this thread's last successful call:
    {"direct": bool, "stream": bool, "record_pass": bool,
    "tensor_cores": bool}."""
    b = _lib().kq_last_kernels()
    return {"direct": bool(b & 1), "stream": bool(b & 2),
            "record_pass": bool(b & 4), "tensor_cores": bool(b & 8)}


def last_launch_count() -> int:
    """Kernel launches enqueued by this thread's last successful call."""
    return int(_lib().kq_last_launch_count())


def set_overlap(enable: bool) -> bool:
    """Let each streaming launch overlap the kernel before it on the stream
    (weights prefetched early; x read and y written only after that kernel
    completes).  Requires that the preceding kernel does not write the
    weights.  Returns the previous setting."""
    return bool(_lib().kq_set_overlap(1 if enable else 0))


def device_error(clear: bool = True) -> bool:
    """True if a kernel on the current device reported an expired wait
    (synchronous read of the device error word)."""
    st = _lib().kq_device_error(1 if clear else 0)
    if st == KQ_ERR_CUDA:
        raise KQError(st, "kq_device_error")
    return st == KQ_ERR_TIMEOUT
