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

ATTN_MASK_NONE = 0
ATTN_MASK_CAUSAL = 1
ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 2
MASKS = {"none": ATTN_MASK_NONE, "causal": ATTN_MASK_CAUSAL,
         "causal_bottom_right": ATTN_MASK_CAUSAL_BOTTOM_RIGHT}

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_MISALIGNED = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5
ATTN_ERR_SCRATCH_TOO_SMALL = 6
STATIC_SCRATCH_BYTES = 16 << 20  # scratch of attn_fwd_kv_static

_lock = threading.Lock()
_lib = None

_FWD_ARGS = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
             ctypes.c_float, ctypes.c_int, ctypes.c_void_p]


_FWD_KV_ARGS = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                ctypes.c_void_p]


_WIN_ARGS = ([ctypes.c_void_p] * 5 + [ctypes.c_int64] * 7 +
             [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p,
              ctypes.c_size_t, ctypes.c_void_p])
ALIGN = {"top_left": 0, "bottom_right": 1}

_BWD_ARGS = ([ctypes.c_void_p] * 9 + [ctypes.c_int64] * 4 +
             [ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
              ctypes.c_void_p])


_BWD_WIN_ARGS = ([ctypes.c_void_p] * 9 + [ctypes.c_int64] * 7 +
                 [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                  ctypes.c_void_p])


_HOST_ARGS = _FWD_ARGS[:12] + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]


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
            lib.attn_fwd_kv.argtypes = _FWD_KV_ARGS
            lib.attn_fwd_kv.restype = ctypes.c_int
            lib.attn_fwd_kv_checked.argtypes = _FWD_KV_ARGS
            lib.attn_fwd_kv_checked.restype = ctypes.c_int
            lib.attn_fwd_kv_workspace_bytes.argtypes = [ctypes.c_int64] * 5
            lib.attn_fwd_kv_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_fwd_kv_static.argtypes = _FWD_KV_ARGS[:13] + [ctypes.c_void_p]
            lib.attn_fwd_kv_static.restype = ctypes.c_int
            lib.attn_fwd_window.argtypes = _WIN_ARGS
            lib.attn_fwd_window.restype = ctypes.c_int
            lib.attn_fwd_window_checked.argtypes = _WIN_ARGS
            lib.attn_fwd_window_checked.restype = ctypes.c_int
            lib.attn_bwd.argtypes = _BWD_ARGS
            lib.attn_bwd.restype = ctypes.c_int
            lib.attn_bwd_checked.argtypes = _BWD_ARGS
            lib.attn_bwd_checked.restype = ctypes.c_int
            lib.attn_bwd_window.argtypes = _BWD_WIN_ARGS
            lib.attn_bwd_window.restype = ctypes.c_int
            lib.attn_bwd_window_checked.argtypes = _BWD_WIN_ARGS
            lib.attn_bwd_window_checked.restype = ctypes.c_int
            lib.attn_bwd_workspace_bytes.argtypes = [ctypes.c_int64] * 4
            lib.attn_bwd_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_fwd_host.argtypes = _HOST_ARGS
            lib.attn_fwd_host.restype = ctypes.c_int
            lib.attn_fwd_host_checked.argtypes = _HOST_ARGS
            lib.attn_fwd_host_checked.restype = ctypes.c_int
            lib.attn_fwd_host_workspace_bytes.argtypes = [ctypes.c_int64] * 4
            lib.attn_fwd_host_workspace_bytes.restype = ctypes.c_size_t
            lib.attn_fwd_host_plan.argtypes = [ctypes.c_int64] * 4 + [ctypes.POINTER(ctypes.c_int64)]
            lib.attn_fwd_host_plan.restype = ctypes.c_int64
            lib.attn_strerror.argtypes = [ctypes.c_int]
            lib.attn_strerror.restype = ctypes.c_char_p
            lib.attn_last_cuda_error.argtypes = []
            lib.attn_last_cuda_error.restype = ctypes.c_int
            lib.attn_device_error_info.argtypes = [ctypes.POINTER(ctypes.c_int32)]
            lib.attn_device_error_info.restype = ctypes.c_int
            lib.attn_probe_tile.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int64, ctypes.c_int,
                                                                    ctypes.c_void_p]
            lib.attn_probe_tile.restype = ctypes.c_int
            lib.attn_probe_wait_timeout.argtypes = [ctypes.c_void_p]
            lib.attn_probe_wait_timeout.restype = ctypes.c_int
            lib.attn_probe_plan_split.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_size_t, ctypes.c_int64,
                                                                        ctypes.POINTER(ctypes.c_int64)]
            lib.attn_probe_plan_split.restype = ctypes.c_int
            lib.attn_probe_plan_decode.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_size_t, ctypes.c_int64,
                                                                          ctypes.POINTER(ctypes.c_int64)]
            lib.attn_probe_plan_decode.restype = ctypes.c_int
            lib.attn_probe_plan_host.argtypes = [ctypes.c_int64] * 3 + [ctypes.POINTER(ctypes.c_int64)]
            lib.attn_probe_plan_host.restype = ctypes.c_int64
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


def attn_fwd_host(q, k, v, o, lse, B, H, N, d, causal, scale, dtype, workspace, workspace_bytes, stream,
                  checked: bool = False) -> int:
    """Raw C call of attn_fwd_host (or its checked form) with integer pointers: q, k, v, o,
    lse in host memory, workspace on the device; returns the attn_status_t."""
    lib = load()
    fn = lib.attn_fwd_host_checked if checked else lib.attn_fwd_host
    return int(fn(q, k, v, o, lse, B, H, N, d, int(bool(causal)), float(scale), int(dtype), workspace,
                  int(workspace_bytes), stream))


def host_workspace_bytes(B, H, N, d) -> int:
    """Device workspace attn_fwd_host needs (0 for sizes it rejects)."""
    return int(load().attn_fwd_host_workspace_bytes(B, H, N, d))


def host_plan(B, H, N, d) -> Tuple[int, int]:
    """(number of chunks, heads per chunk) of attn_fwd_host; (0, 0) for rejected sizes."""
    h = ctypes.c_int64(0)
    n = int(load().attn_fwd_host_plan(B, H, N, d, ctypes.byref(h)))
    return n, int(h.value) if n else 0


def plan_split_for(BH, Nq, Nk, d, ws_bytes, sms) -> Tuple[int, int, int]:
    """(key ranges, key tiles per range, workspace bytes) of attn_fwd_kv's split of the
    keys on a GPU with `sms` SMs (test hook)."""
    out = (ctypes.c_int64 * 3)()
    st = load().attn_probe_plan_split(BH, Nq, Nk, d, ws_bytes, sms, out)
    if st != ATTN_OK:
        raise AttnError(st, f"attn_probe_plan_split: {strerror(st)}")
    return int(out[0]), int(out[1]), int(out[2])


def plan_decode_for(BH, Nq, Nk, d, ws_bytes, sms) -> Tuple[int, int, int, int]:
    """(key ranges per head, keys per range, CTAs, workspace bytes) of the streaming
    decode kernel on a GPU with `sms` SMs (test hook)."""
    out = (ctypes.c_int64 * 4)()
    st = load().attn_probe_plan_decode(BH, Nq, Nk, d, ws_bytes, sms, out)
    if st != ATTN_OK:
        raise AttnError(st, f"attn_probe_plan_decode: {strerror(st)}")
    return int(out[0]), int(out[1]), int(out[2]), int(out[3])


def plan_host_for(BH, N, sms) -> Tuple[int, int]:
    """(chunks, heads per chunk) of attn_fwd_host on a GPU with `sms` SMs (test hook)."""
    h = ctypes.c_int64(0)
    n = int(load().attn_probe_plan_host(BH, N, sms, ctypes.byref(h)))
    return n, int(h.value) if n else 0


def attn_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, workspace, workspace_bytes,
                stream, checked: bool = False) -> int:
    """Raw C call of attn_fwd_kv (or attn_fwd_kv_checked); returns the attn_status_t."""
    lib = load()
    fn = lib.attn_fwd_kv_checked if checked else lib.attn_fwd_kv
    return int(fn(q, k, v, o, lse, B, H, Nq, Nk, d, int(mask), float(scale), int(dtype), workspace,
                  int(workspace_bytes), stream))


def workspace_bytes(B, H, Nq, Nk, d) -> int:
    """Workspace size for attn_fwd_kv's full split of the keys (0: never splits)."""
    return int(load().attn_fwd_kv_workspace_bytes(B, H, Nq, Nk, d))


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


def fwd_host(q, k, v, causal: bool = False, scale: Optional[float] = None, out=None, lse=None,
             workspace=None, device=None, stream=None, checked: bool = False) -> Tuple[object, object]:
    """Attention forward of CPU tensors q, k, v [B, H, N, d] (fp16/bf16, contiguous) through
    attn_fwd_host: the copies to and from the GPU and the kernels run pipelined by chunks of
    heads. Returns (o, lse) as CPU tensors (page-locked unless ``out``/``lse`` are given),
    complete on return: the stream is synchronised. ``workspace`` is a CUDA uint8 tensor of
    :func:`host_workspace_bytes` bytes (allocated here when not given) on ``device``.

    q = k = v = None reuses the inputs an earlier call staged in ``workspace`` (then ``out``
    gives the shape and dtype, and ``lse`` and ``workspace`` must be given too)."""
    import torch
    if q is None and k is None and v is None:
        if out is None or lse is None or workspace is None:
            raise ValueError("reusing staged inputs needs out, lse and workspace")
        B, H, N, d = out.shape
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        if stream is None:
            stream = torch.cuda.current_stream(workspace.device)
        st = attn_fwd_host(None, None, None, out.data_ptr(), lse.data_ptr(), B, H, N, d, causal, scale,
                           _dtype_code(out), workspace.data_ptr(), workspace.numel(), stream.cuda_stream,
                           checked=checked)
        _check(st, "attn_fwd_host")
        stream.synchronize()
        return out, lse
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CPU tensors")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    if workspace is None:
        dev = torch.device("cuda") if device is None else torch.device(device)
        workspace = torch.empty((host_workspace_bytes(B, H, N, d),), dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    st = attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
                       causal, scale, _dtype_code(q), workspace.data_ptr(), workspace.numel(), stream.cuda_stream,
                       checked=checked)
    _check(st, "attn_fwd_host")
    stream.synchronize()
    return out, lse


def fwd_kv(q, k, v, mask: str = "none", scale: Optional[float] = None, out=None, lse=None,
           workspace=None, stream=None, checked: bool = False) -> Tuple[object, object]:
    """Attention forward of q [B, H, Nq, d] against k, v [B, H, Nk, d] (CUDA, fp16/bf16,
    contiguous), e.g. one KV-cache decode step.

    ``mask`` is "none", "causal" (row i sees keys j <= i) or "causal_bottom_right"
    (row i sees keys j <= i + Nk - Nq). ``workspace`` is a CUDA uint8 tensor for the
    split of the keys; by default one of :func:`workspace_bytes` bytes is allocated
    here (pass ``workspace=False`` for none). Returns (o like q, lse fp32 [B, H, Nq]).
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] must agree on B, H and d")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    if mask not in MASKS:
        raise ValueError(f"mask must be one of {sorted(MASKS)}")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = workspace_bytes(B, H, Nq, Nk, d)
        workspace = torch.empty((n,), dtype=torch.uint8, device=q.device) if n else False
    ws_ptr, ws_n = (workspace.data_ptr(), workspace.numel()) if workspace is not False else (None, 0)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H,
                     Nq, Nk, d, MASKS[mask], scale, _dtype_code(q), ws_ptr, ws_n, stream.cuda_stream,
                     checked=checked)
    _check(st, "attn_fwd_kv")
    return out, lse


def attn_fwd_window(q, k, v, o, lse, B, H, Nq, Nk, d, window_left, window_right, kv_lens, align, scale,
                    dtype, workspace, workspace_bytes, stream, checked: bool = False) -> int:
    """Raw C call of attn_fwd_window (or its checked form); returns the attn_status_t."""
    lib = load()
    fn = lib.attn_fwd_window_checked if checked else lib.attn_fwd_window
    return int(fn(q, k, v, o, lse, B, H, Nq, Nk, d, int(window_left), int(window_right), kv_lens,
                  int(align), float(scale), int(dtype), workspace, int(workspace_bytes), stream))


def fwd_window(q, k, v, window=(-1, -1), kv_lens=None, align: str = "top_left",
               scale: Optional[float] = None, out=None, lse=None, workspace=None, stream=None,
               checked: bool = False):
    """Forward of q [B,H,Nq,d] against k, v [B,H,Nk,d] with a sliding window
    ``(left, right)`` around the diagonal (negative: unbounded; right = 0 is causal) and
    optional per-batch valid key counts ``kv_lens`` (CUDA int32 [B]). Rows that see no
    key get O = 0 and LSE = -inf. Returns (o, lse)."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] must agree on B, H and d")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if kv_lens is not None:
        if kv_lens.dtype != torch.int32 or kv_lens.shape != (B,) or not kv_lens.is_cuda:
            raise ValueError("kv_lens must be a CUDA int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        n = workspace_bytes(B, H, Nq, Nk, d)
        workspace = torch.empty((n,), dtype=torch.uint8, device=q.device) if n else False
    ws_ptr, ws_n = (workspace.data_ptr(), workspace.numel()) if workspace is not False else (None, 0)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_fwd_window(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Nq,
                         Nk, d, window[0], window[1], kv_lens.data_ptr() if kv_lens is not None else None,
                         ALIGN[align], scale, _dtype_code(q), ws_ptr, ws_n, stream.cuda_stream, checked=checked)
    _check(st, "attn_fwd_window")
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, dtype, workspace,
             workspace_bytes, stream, checked: bool = False) -> int:
    """Raw C call of attn_bwd (or attn_bwd_checked); returns the attn_status_t."""
    lib = load()
    fn = lib.attn_bwd_checked if checked else lib.attn_bwd
    return int(fn(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, int(bool(causal)), float(scale),
                  int(dtype), workspace, int(workspace_bytes), stream))


def bwd_workspace_bytes(B, H, N, d) -> int:
    """Workspace attn_bwd needs for these sizes (0 for sizes it rejects)."""
    return int(load().attn_bwd_workspace_bytes(B, H, N, d))


def bwd(q, k, v, o, lse, dout, causal: bool = False, scale: Optional[float] = None, dq=None,
        dk=None, dv=None, workspace=None, stream=None, checked: bool = False):
    """Gradients (dq, dk, dv) of sum(dout * o) for o, lse = fwd(q, k, v, causal, scale).

    All tensors contiguous CUDA [B, H, N, d] of one 16-bit dtype; lse fp32 [B, H, N].
    ``workspace`` (a CUDA uint8 tensor of :func:`bwd_workspace_bytes` bytes) is
    allocated here when not given.
    """
    import torch
    for t in (q, k, v, o, dout):
        if t.dim() != 4 or t.shape != q.shape:
            raise ValueError("q, k, v, o and dout must all be [B, H, N, d]")
        if t.dtype != q.dtype:
            raise TypeError("q, k, v, o and dout must share one dtype")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    B, H, N, d = q.shape
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if workspace is None:
        workspace = torch.empty((max(bwd_workspace_bytes(B, H, N, d), 16),), dtype=torch.uint8,
                                device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                  dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, causal,
                  scale, _dtype_code(q), workspace.data_ptr(), workspace.numel(), stream.cuda_stream,
                  checked=checked)
    _check(st, "attn_bwd")
    return dq, dk, dv


def bwd_window(q, k, v, o, lse, dout, window=(-1, -1), kv_lens=None, align: str = "top_left",
               scale: Optional[float] = None, workspace=None, stream=None, checked: bool = False):
    """Gradients (dq [B,H,Nq,d], dk, dv [B,H,Nk,d]) of sum(dout * o) for
    o, lse = fwd_window(q, k, v, window, kv_lens, align, scale)."""
    import torch
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    for t, n in ((q, Nq), (o, Nq), (dout, Nq), (k, Nk), (v, Nk)):
        if t.dim() != 4 or t.shape != (B, H, n, d) or t.dtype != q.dtype:
            raise ValueError("q, o, dout [B,H,Nq,d] and k, v [B,H,Nk,d] of one dtype")
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("inputs must be contiguous CUDA tensors")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    if kv_lens is not None and (kv_lens.dtype != torch.int32 or kv_lens.shape != (B,) or not kv_lens.is_cuda):
        raise ValueError("kv_lens must be a CUDA int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    if workspace is None:
        workspace = torch.empty((max(bwd_workspace_bytes(B, H, Nq, d), 16),), dtype=torch.uint8,
                                device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    fn = load().attn_bwd_window_checked if checked else load().attn_bwd_window
    st = int(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d, int(window[0]), int(window[1]),
                kv_lens.data_ptr() if kv_lens is not None else None, ALIGN[align], float(scale), _dtype_code(q),
                workspace.data_ptr(), workspace.numel(), stream.cuda_stream))
    _check(st, "attn_bwd_window")
    return dq, dk, dv


def attn_fwd_kv_static(q, k, v, o, lse, B, H, Nq, Nk, d, mask, scale, dtype, stream) -> int:
    """Raw C call of attn_fwd_kv_static (integer pointers); returns the attn_status_t."""
    return int(load().attn_fwd_kv_static(q, k, v, o, lse, B, H, Nq, Nk, d, int(mask), float(scale),
                                         int(dtype), stream))


def fwd_kv_static(q, k, v, out, lse, mask: str = "none", scale: Optional[float] = None,
                  stream=None) -> Tuple[object, object]:
    """:func:`fwd_kv` through attn_fwd_kv_static: nothing is allocated on this path, so
    the caller passes ``out`` (like q) and ``lse`` (fp32 [B, H, Nq]). Calls on one device
    share the library's static scratch and must not overlap in time."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != q.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] must agree on B, H and d")
    if not (q.dtype == k.dtype == v.dtype == out.dtype):
        raise TypeError("q, k, v and out must share one dtype")
    if out.shape != q.shape or lse.shape != q.shape[:3] or lse.dtype != torch.float32:
        raise ValueError("out must be like q and lse fp32 [B, H, Nq]")
    for t in (q, k, v, out, lse):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v, out and lse must be contiguous CUDA tensors")
    if mask not in MASKS:
        raise ValueError(f"mask must be one of {sorted(MASKS)}")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_fwd_kv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                            B, H, Nq, Nk, d, MASKS[mask], scale, _dtype_code(q), stream.cuda_stream)
    _check(st, "attn_fwd_kv_static")
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
