"""fp64 CPU oracle for the exact scaled-dot-product attention forward and backward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the CUDA path neither
imports it nor shares code with it.

Three functions compute the same thing three ways, so that each checks the others:

* :func:`attn_fwd` / :func:`attn_fwd_rows` -- the plain definition, per query row,
  in C (``attn_oracle.c``, fp64, OpenMP). This is the oracle proper.
* :func:`attn_fwd_materialised` -- numpy fp64, the whole N x N score matrix at once,
  as in "Programming an attention kernel in Triton", Kernel 4 (scores, mask with
  -inf, softmax over keys, weights times V). For small N only.
* :func:`attn_fwd_online` -- numpy fp64, the tiled online-softmax forward in the
  order of "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel" (the
  profile-driven FlashAttention-2 page): raw scores per key tile, mask, running
  max kept in log2 units of the scaled scores (Round 4 / exp2), rescale factor
  alpha, running sum l, unnormalised O, and at the end O / l and
  L = (m + log2 l) ln 2. An optional threshold ``tau`` keeps a stale maximum
  until the row maximum grows by more than ``tau`` (log2 units); the result is
  the same because O and l always share the maximum they were scaled by.

The backward (the gradients of sum(dO * O)) has the same pair: :func:`attn_bwd`
in C, the chain rule through the definition per query row, and
:func:`attn_bwd_materialised` in numpy on whole matrices. The forward-only
variants :func:`attn_fwd_qk` (Nq query rows against Nk keys) follow the forward.

Inputs are 16-bit (or fp32/fp64) tensors/arrays of shape [B, H, N, d]; they are
upcast exactly to fp64 before any arithmetic. Outputs are fp64: O [B, H, N, d]
and LSE [B, H, N] (natural log).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_DP = ctypes.POINTER(ctypes.c_double)
_I64P = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``_build/liboracle.so`` (gcc, fp64, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attn_fwd.argtypes = [_DP, _DP, _DP, _DP, _DP, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int, ctypes.c_double]
            lib.oracle_attn_fwd.restype = ctypes.c_int
            lib.oracle_attn_rows.argtypes = [_DP, _DP, _DP, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                                             _I64P, ctypes.c_int64, _DP, _DP]
            lib.oracle_attn_rows.restype = ctypes.c_int
            lib.oracle_attn_fwd_qk.argtypes = [_DP, _DP, _DP, _DP, _DP, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int, ctypes.c_double]
            lib.oracle_attn_fwd_qk.restype = ctypes.c_int
            lib.oracle_attn_fwd_window.argtypes = [_DP, _DP, _DP, _DP, _DP] + [ctypes.c_int64] * 7 + [
                _I64P, ctypes.c_int, ctypes.c_double]
            lib.oracle_attn_fwd_window.restype = ctypes.c_int
            lib.oracle_attn_bwd.argtypes = [_DP, _DP, _DP, _DP, _DP, _DP, _DP, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_double]
            lib.oracle_attn_bwd.restype = ctypes.c_int
            lib.oracle_attn_bwd_window.argtypes = [_DP] * 7 + [ctypes.c_int64] * 7 + [
                _I64P, ctypes.c_int, ctypes.c_double]
            lib.oracle_attn_bwd_window.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the C oracle uses."""
    return int(_load().oracle_num_threads())


def to_f64(x) -> np.ndarray:
    """Exact upcast of a torch tensor (fp16/bf16/fp32/fp64) or numpy array to fp64."""
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    import torch  # plain CPU conversion only
    return np.ascontiguousarray(x.detach().to("cpu").to(torch.float64).numpy())


def default_scale(d: int) -> float:
    """1/sqrt(d), the softmax scale of the workloads."""
    return 1.0 / math.sqrt(d)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_DP)


def attn_fwd(q, k, v, causal: bool, scale: float | None = None):
    """Plain-definition oracle (C, fp64). Returns (O [B,H,N,d], LSE [B,H,N])."""
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, d = q64.shape
    if k64.shape != q64.shape or v64.shape != q64.shape:
        raise ValueError("q, k, v must share the shape [B, H, N, d]")
    scale = default_scale(d) if scale is None else float(scale)
    o = np.empty_like(q64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attn_fwd(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(o), _ptr(lse),
                                 B, H, N, d, int(bool(causal)), scale)
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd failed with code {rc}")
    return o, lse


_ALIGN = {"bottom_right": 1, "top_left": 2}


def attn_fwd_qk(q, k, v, causal: bool, scale: float | None = None, align: str = "bottom_right"):
    """Nq query rows [B,H,Nq,d] against Nk keys [B,H,Nk,d] (C, fp64).

    Under the causal mask with ``align="bottom_right"`` the query rows are the last
    Nq positions of the Nk-long sequence: row i sees keys j <= i + Nk - Nq (a
    KV-cache decode step). With ``align="top_left"`` row i sees keys j <= i, the
    k_pos <= q_pos test of the profile-driven FlashAttention-2 page ("Round 4 /
    Causal tile-skipping") applied to its separate N_QUERIES and N_KEYS. A row with
    no visible key gets O = 0 and LSE = -inf. Returns (O [B,H,Nq,d], LSE [B,H,Nq]).
    """
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, Nq, d = q64.shape
    Bk, Hk, Nk, dk = k64.shape
    if (Bk, Hk, dk) != (B, H, d) or v64.shape != k64.shape:
        raise ValueError("q [B,H,Nq,d], k and v [B,H,Nk,d] must agree on B, H, d")
    scale = default_scale(d) if scale is None else float(scale)
    o = np.empty_like(q64)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    rc = _load().oracle_attn_fwd_qk(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(o), _ptr(lse),
                                    B * H, Nq, Nk, d, _ALIGN[align] if causal else 0, scale)
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_qk failed with code {rc}")
    return o, lse


def attn_fwd_qk_materialised(q, k, v, causal: bool, scale: float | None = None,
                             align: str = "bottom_right"):
    """numpy fp64 twin of :func:`attn_fwd_qk` with the whole Nq x Nk score matrix."""
    shift = {"bottom_right": None, "top_left": 0}[align]
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, Nq, d = q64.shape
    Nk = k64.shape[2]
    scale = default_scale(d) if scale is None else float(scale)
    s = scale * np.einsum("bhid,bhjd->bhij", q64, k64)
    keep = np.ones((Nq, Nk), dtype=bool)
    if causal:
        keep = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq if shift is None else shift)
    s = np.where(keep, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe)
    l = e.sum(axis=-1, keepdims=True)
    o = np.einsum("bhij,bhjd->bhid", e, v64) / np.where(empty, 1.0, l)
    lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))[..., 0]
    return o, lse


def attn_fwd_rows(q, k, v, causal: bool, rows, scale: float | None = None):
    """Oracle outputs for selected rows only.

    ``rows`` holds flat row indices ``(b*H + h)*N + i``. Returns (O [R,d], LSE [R]).
    """
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, d = q64.shape
    scale = default_scale(d) if scale is None else float(scale)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.empty((r.size, d), dtype=np.float64)
    lse = np.empty((r.size,), dtype=np.float64)
    rc = _load().oracle_attn_rows(_ptr(q64), _ptr(k64), _ptr(v64), B * H, N, d,
                                  int(bool(causal)), scale, r.ctypes.data_as(_I64P), r.size,
                                  _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_attn_rows failed with code {rc}")
    return o, lse


def attn_fwd_materialised(q, k, v, causal: bool, scale: float | None = None):
    """numpy fp64 twin that builds the whole N x N score matrix (small N only)."""
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, d = q64.shape
    scale = default_scale(d) if scale is None else float(scale)
    s = scale * np.einsum("bhid,bhjd->bhij", q64, k64)
    if causal:
        keep = np.tril(np.ones((N, N), dtype=bool))
        s = np.where(keep, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    o = np.einsum("bhij,bhjd->bhid", e, v64) / l
    lse = (m + np.log(l))[..., 0]
    return o, lse


def attn_fwd_online(q, k, v, causal: bool, scale: float | None = None,
                    block: int = 128, tau: float = 0.0):
    """Tiled online-softmax forward in fp64 (see the module docstring)."""
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, N, d = q64.shape
    scale = default_scale(d) if scale is None else float(scale)
    if block < 1:
        raise ValueError("block must be >= 1")
    qk_scale = scale * math.log2(math.e)
    q_pos = np.arange(N)[:, None]
    o_out = np.empty_like(q64)
    lse_out = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            Q, K, V = q64[b, h], k64[b, h], v64[b, h]
            m = np.full((N, 1), -np.inf)
            l = np.zeros((N, 1))
            acc = np.zeros((N, d))
            for start in range(0, N, block):
                stop = min(start + block, N)
                S = Q @ K[start:stop].T                      # raw scores, unscaled
                k_pos = np.arange(start, stop)[None, :]
                keep = np.ones_like(S, dtype=bool)
                if causal:
                    keep &= k_pos <= q_pos
                S = np.where(keep, S, -np.inf)
                m_new = np.maximum(m, S.max(axis=1, keepdims=True) * qk_scale)
                if tau > 0.0:
                    # keep the stale maximum while it is within tau of the new one
                    stale_ok = np.isfinite(m) & (m_new - m <= tau)
                    m_new = np.where(stale_ok, m, m_new)
                m_use = np.where(np.isneginf(m_new), 0.0, m_new)
                P = np.exp2(S * qk_scale - m_use)
                alpha = np.exp2(m - m_use)
                l = alpha * l + P.sum(axis=1, keepdims=True)
                acc = alpha * acc + P @ V[start:stop]
                m = m_new
            o_out[b, h] = acc / l
            lse_out[b, h] = ((m + np.log2(l)) * math.log(2.0))[:, 0]
    return o_out, lse_out


def attn_bwd(q, k, v, dout, causal: bool, scale: float | None = None):
    """Gradients (dQ, dK, dV) of sum(dO * O) for O = attention(Q, K, V) (C, fp64).

    The chain rule through the definition, per query row: P = exp(s - LSE),
    dV += P^T dO, dP = dO V^T, D = rowsum(P * dP), dS = P * (dP - D),
    dQ = scale dS K, dK = scale dS^T Q. All inputs [B,H,N,d]; returns three
    float64 arrays of that shape.
    """
    q64, k64, v64, g64 = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, H, N, d = q64.shape
    for t in (k64, v64, g64):
        if t.shape != q64.shape:
            raise ValueError("q, k, v and dout must have the same shape")
    scale = default_scale(d) if scale is None else float(scale)
    dq, dk, dv = (np.empty_like(q64) for _ in range(3))
    rc = _load().oracle_attn_bwd(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B * H, N, d, int(bool(causal)), scale)
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd failed with code {rc}")
    return dq, dk, dv


def attn_bwd_materialised(q, k, v, dout, causal: bool, scale: float | None = None):
    """numpy fp64 twin of :func:`attn_bwd` on whole N x N matrices.

    Returns a dict with dq, dk, dv and the intermediates p (softmax weights), dp
    (dO V^T), ds (P * (dP - D)) and D, all float64.
    """
    q64, k64, v64, g64 = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    N, d = q64.shape[2], q64.shape[3]
    scale = default_scale(d) if scale is None else float(scale)
    s = scale * np.einsum("bhid,bhjd->bhij", q64, k64)
    if causal:
        s = np.where(np.tril(np.ones((N, N), dtype=bool)), s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    p = e / e.sum(axis=-1, keepdims=True)
    dp = np.einsum("bhid,bhjd->bhij", g64, v64)
    D = (p * dp).sum(axis=-1, keepdims=True)
    ds = p * (dp - D)
    return {
        "dq": scale * np.einsum("bhij,bhjd->bhid", ds, k64),
        "dk": scale * np.einsum("bhij,bhid->bhjd", ds, q64),
        "dv": np.einsum("bhij,bhid->bhjd", p, g64),
        "p": p, "dp": dp, "ds": ds, "D": D[..., 0],
    }


def attn_fwd_window(q, k, v, left: int = -1, right: int = -1, kv_lens=None, align: str = "top_left",
                    scale: float | None = None):
    """Nq query rows [B,H,Nq,d] against Nk keys [B,H,Nk,d] with a sliding window and key
    padding (C, fp64).

    Batch element b has ``kv_lens[b]`` valid keys (None: all). Row i's diagonal is key
    i + off_b with off_b = 0 (``align="top_left"``) or kv_lens[b] - Nq
    (``"bottom_right"``); it sees valid keys diag - left <= j <= diag + right, a negative
    bound meaning unbounded on that side (right = 0 is the causal mask). Rows that see no
    key get O = 0 and LSE = -inf. Returns (O [B,H,Nq,d], LSE [B,H,Nq]).
    """
    q64, k64, v64 = to_f64(q), to_f64(k), to_f64(v)
    B, H, Nq, d = q64.shape
    Nk = k64.shape[2]
    if k64.shape != (B, H, Nk, d) or v64.shape != k64.shape:
        raise ValueError("q [B,H,Nq,d], k and v [B,H,Nk,d] must agree on B, H, d")
    scale = default_scale(d) if scale is None else float(scale)
    lens = None
    if kv_lens is not None:
        lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int64).reshape(B))
    o = np.empty_like(q64)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    rc = _load().oracle_attn_fwd_window(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(o), _ptr(lse), B, H, Nq,
                                        Nk, d, int(left), int(right),
                                        lens.ctypes.data_as(_I64P) if lens is not None else None,
                                        {"top_left": 0, "bottom_right": 1}[align], scale)
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_window failed with code {rc}")
    return o, lse


def window_mask(B, Nq, Nk, left=-1, right=-1, kv_lens=None, align="top_left"):
    """Boolean [B, Nq, Nk] visibility of :func:`attn_fwd_window`, spelled out in numpy."""
    lens = np.full(B, Nk) if kv_lens is None else np.asarray(kv_lens).reshape(B)
    i = np.arange(Nq)[None, :, None]
    j = np.arange(Nk)[None, None, :]
    n = lens[:, None, None]
    diag = i + (n - Nq if align == "bottom_right" else 0)
    keep = j < n
    if left >= 0:
        keep = keep & (j >= diag - left)
    if right >= 0:
        keep = keep & (j <= diag + right)
    return keep


def attn_bwd_window(q, k, v, dout, left: int = -1, right: int = -1, kv_lens=None,
                    align: str = "top_left", scale: float | None = None):
    """Gradients (dQ [B,H,Nq,d], dK, dV [B,H,Nk,d]) of sum(dO * O) for O of
    :func:`attn_fwd_window` (C, fp64): each query row over exactly the keys it sees."""
    q64, k64, v64, g64 = to_f64(q), to_f64(k), to_f64(v), to_f64(dout)
    B, H, Nq, d = q64.shape
    Nk = k64.shape[2]
    if k64.shape != (B, H, Nk, d) or v64.shape != k64.shape or g64.shape != q64.shape:
        raise ValueError("q, dout [B,H,Nq,d] and k, v [B,H,Nk,d] must agree")
    scale = default_scale(d) if scale is None else float(scale)
    lens = None
    if kv_lens is not None:
        lens = np.ascontiguousarray(np.asarray(kv_lens, dtype=np.int64).reshape(B))
    dq, dk, dv = np.empty_like(q64), np.empty_like(k64), np.empty_like(k64)
    rc = _load().oracle_attn_bwd_window(_ptr(q64), _ptr(k64), _ptr(v64), _ptr(g64), _ptr(dq), _ptr(dk),
                                        _ptr(dv), B, H, Nq, Nk, d, int(left), int(right),
                                        lens.ctypes.data_as(_I64P) if lens is not None else None,
                                        {"top_left": 0, "bottom_right": 1}[align], scale)
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd_window failed with code {rc}")
    return dq, dk, dv
