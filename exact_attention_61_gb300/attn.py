"""Thin ctypes binding of the C ABI in ``include/attn.h`` (argument marshalling only).

Every step of the forward runs in the CUDA kernels of ``libattn.so``; this module
only turns torch tensors into pointers and sizes. There is no fallback: if the
library is missing or the call fails, it raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn.so")

ATTN_FP16 = 0
ATTN_BF16 = 1

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5

_lock = threading.Lock()
_lib = None

_FWD_ARGS = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
             ctypes.c_float, ctypes.c_int, ctypes.c_void_p]


class AttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def load(path: str = LIB_PATH):
    """Load ``libattn.so`` (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(path)
            lib.attn_fwd.argtypes = _FWD_ARGS
            lib.attn_fwd.restype = ctypes.c_int
            lib.attn_fwd_checked.argtypes = _FWD_ARGS
            lib.attn_fwd_checked.restype = ctypes.c_int
            lib.attn_strerror.argtypes = [ctypes.c_int]
            lib.attn_strerror.restype = ctypes.c_char_p
            lib.attn_last_cuda_error.argtypes = []
            lib.attn_last_cuda_error.restype = ctypes.c_int
            lib.attn_device_error_info.argtypes = [ctypes.POINTER(ctypes.c_int32)]
            lib.attn_device_error_info.restype = ctypes.c_int
            lib.attn_probe_tile.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int64, ctypes.c_int,
                                                                    ctypes.c_void_p]
            lib.attn_probe_tile.restype = ctypes.c_int
            _lib = lib
    return _lib


def strerror(status: int) -> str:
    return load().attn_strerror(int(status)).decode()


def last_cuda_error() -> int:
    return int(load().attn_last_cuda_error())


def device_error_info():
    info = (ctypes.c_int32 * 4)()
    st = load().attn_device_error_info(info)
    if st != ATTN_OK:
        raise AttnError(st, strerror(st))
    return list(info)


def _check(status: int, what: str):
    if status != ATTN_OK:
        extra = ""
        if status == ATTN_ERR_CUDA:
            extra = f" (cuda error {last_cuda_error()})"
        elif status == ATTN_ERR_TIMEOUT:
            extra = f" (device record {device_error_info()})"
        raise AttnError(status, f"{what}: {strerror(status)}{extra}")


def attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, stream) -> int:
    """Raw C call with integer pointers; returns the attn_status_t."""
    return int(load().attn_fwd(q, k, v, o, lse, B, H, N, d, int(bool(causal)), float(scale),
                               int(dtype), stream))


def attn_fwd_checked(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, stream) -> int:
    return int(load().attn_fwd_checked(q, k, v, o, lse, B, H, N, d, int(bool(causal)),
                                       float(scale), int(dtype), stream))


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return ATTN_FP16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: expected float16 or bfloat16")


def fwd(q, k, v, causal: bool = False, scale: Optional[float] = None, out=None, lse=None,
        stream=None, checked: bool = False) -> Tuple[object, object]:
    """Attention forward on CUDA tensors [B, H, N, d] (fp16/bf16, contiguous).

    Returns (o, lse): o like q, lse fp32 [B, H, N] (natural log). ``out``/``lse``
    may be given to write into existing buffers. Runs on ``stream`` (default: the
    current torch stream).
    """
    import torch
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    call = attn_fwd_checked if checked else attn_fwd
    st = call(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N,
              d, causal, scale, _dtype_code(q), stream.cuda_stream)
    _check(st, "attn_fwd")
    return out, lse


def probe_tile(q, k, v, p, stream=None):
    """One-tile tensor-core probe: returns (S = q k^T, O = p v) as fp32 CUDA tensors."""
    import torch
    d = q.shape[-1]
    s_out = torch.empty((128, 128), dtype=torch.float32, device=q.device)
    o_out = torch.empty((128, d), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = load().attn_probe_tile(q.data_ptr(), k.data_ptr(), v.data_ptr(), p.data_ptr(),
                                s_out.data_ptr(), o_out.data_ptr(), d, _dtype_code(q),
                                stream.cuda_stream)
    _check(st, "attn_probe_tile")
    return s_out, o_out
