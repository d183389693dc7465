"""Parity of the windowed / padded / Nq != Nk backward (attn_bwd_window, through the C
ABI) with the fp64 oracle (oracle.attn_bwd_window), element by element within the
rounding bound of oracle/bwd_bound.py (P, dS, D and the outputs rounded once), with
P and dS materialised under the same visibility mask. Rows that see no key must give
dQ = 0 exactly and padded keys dK = dV = 0 exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gen import make_qkv_kv
from oracle import bwd_bound

DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _masked_p_ds(q64, k64, v64, do64, keep, scale):
    s = scale * np.einsum("bhid,bhjd->bhij", q64, k64)
    s = np.where(keep[:, None], s, -np.inf)
    m = s.max(-1, keepdims=True)
    has = np.isfinite(m)
    e = np.where(has, np.exp(s - np.where(has, m, 0.0)), 0.0)
    p = e / np.maximum(e.sum(-1, keepdims=True), 1e-300)
    dp = np.einsum("bhid,bhjd->bhij", do64, v64)
    D = (p * dp).sum(-1, keepdims=True)
    return p, p * (dp - D)


def _case(attn, B, H, Nq, Nk, d, dtype, window, lens, align, seed, e2e=False):
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, dtype, seed)
    do = make_qkv_kv(B, H, Nq, 1, d, dtype, seed + 7919)[0]
    scale = 1.0 / math.sqrt(d)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    gq, gk, gv, gdo = (t.cuda() for t in (q, k, v, do))
    o_ref, lse_ref = oracle.attn_fwd_window(q, k, v, window[0], window[1], lens, align, scale)
    if e2e:
        o, lse = attn.fwd_window(gq, gk, gv, window=window, kv_lens=kl, align=align, scale=scale, checked=True)
    else:
        o = torch.from_numpy(o_ref).to(DT[dtype]).cuda()
        lse = torch.from_numpy(lse_ref).to(torch.float32).cuda()
    dq, dk, dv = attn.bwd_window(gq, gk, gv, o, lse, gdo, window=window, kv_lens=kl, align=align, scale=scale,
                                 checked=True)
    ref = dict(zip(("dq", "dk", "dv"), oracle.attn_bwd_window(q, k, v, do, window[0], window[1], lens, align,
                                                              scale)))
    q64, k64, v64, do64 = (oracle.to_f64(t) for t in (q, k, v, do))
    keep = oracle.window_mask(B, Nq, Nk, window[0], window[1], lens, align)
    p, ds = _masked_p_ds(q64, k64, v64, do64, keep, scale)
    o_used = o.to(torch.float64).cpu().numpy()
    dD = bwd_bound.d_error(do64, o_used, o_ref, bwd_bound.U[dtype])
    bnd = bwd_bound.bounds(ref, {"p": p, "ds": ds}, q64, k64, do64, dD, scale, dtype, max(Nq, Nk))
    name = f"B{B}H{H}q{Nq}k{Nk}d{d}{dtype} w{window} lens{lens} {align}{' e2e' if e2e else ''}"
    got = {"dq": dq, "dk": dk, "dv": dv}
    ok, msg = bwd_bound.check({key: t.to(torch.float64).cpu().numpy() for key, t in got.items()}, ref, bnd)
    assert ok, f"{name}: {msg}"
    # exact zeros: rows with no key, padded keys
    no_key = ~keep.any(-1)  # [B, Nq]
    rows = np.broadcast_to(no_key[:, None, :], (B, H, Nq))
    assert (got["dq"].float().cpu().numpy()[rows] == 0).all(), name
    if lens is not None:
        for b, n in enumerate(lens):
            assert (got["dk"][b, :, n:] == 0).all() and (got["dv"][b, :, n:] == 0).all(), name


@pytest.mark.gpu
@pytest.mark.parametrize("window", [(127, 0), (128, 0), (300, 0), (64, 64), (0, 0), (200, -1), (-1, 50)], ids=str)
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "fp16")])
def test_square_windows(cuda_lib, window, d, dtype):
    _case(cuda_lib, 1, 3, 700, 700, d, dtype, window, None, "top_left", seed=64000 + window[0] + d)


@pytest.mark.gpu
@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (100, 0)], ids=str)
@pytest.mark.parametrize("align", ["top_left", "bottom_right"])
def test_padding(cuda_lib, window, align):
    _case(cuda_lib, 4, 2, 600, 600, 64, "bf16", window, [600, 257, 1, 0], align, seed=64100 + len(align))


@pytest.mark.gpu
@pytest.mark.parametrize("Nq,Nk,window,align", [
    (300, 1000, (-1, 0), "bottom_right"),
    (1000, 300, (-1, 0), "bottom_right"),   # the first 700 rows see no key
    (257, 700, (-1, -1), "top_left"),
    (700, 257, (100, 0), "top_left"),
    (64, 2000, (500, 0), "bottom_right"),
    (129, 1500, (-1, 0), "top_left"),
])
@pytest.mark.parametrize("d", [64, 128])
def test_cross_lengths(cuda_lib, Nq, Nk, window, align, d):
    _case(cuda_lib, 2, 2, Nq, Nk, d, "bf16", window, [Nk, max(1, Nk // 2)], align, seed=64200 + Nq + Nk + d)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_end_to_end_with_cuda_forward(cuda_lib, d):
    _case(cuda_lib, 2, 2, 500, 900, d, "bf16", (200, 0), [900, 450], "bottom_right", seed=64300 + d, e2e=True)


@pytest.mark.gpu
def test_plain_masks_match_attn_bwd_bitwise(cuda_lib):
    """Without padding or a window and with Nq = Nk, attn_bwd_window runs the plain kernel."""
    q, k, v = (t.cuda() for t in make_qkv_kv(2, 4, 800, 800, 64, "bf16", 64400))
    do = make_qkv_kv(2, 4, 800, 1, 64, "bf16", 64401)[0].cuda()
    for causal in (False, True):
        o, lse = cuda_lib.fwd(q, k, v, causal=causal, checked=True)
        a = cuda_lib.bwd(q, k, v, o, lse, do, causal=causal, checked=True)
        b = cuda_lib.bwd_window(q, k, v, o, lse, do, window=(-1, 0 if causal else -1), checked=True)
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
        assert (a[0].float() - b[0].float()).abs().max().item() <= 2 * 2.0 ** -8 * a[0].float().abs().max().item()
