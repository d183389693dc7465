"""Parity of the Nq-against-Nk forward (attn_fwd_kv, through the C ABI) with the fp64
oracle: KV-cache decode steps (few query rows, long key cache, keys split over CTAs
and merged), cross lengths in both directions with ragged tails, the two causal
alignments, and rows that see no key.

Tolerances as for the square forward: O max-abs 4e-3 (fp16) / 3.2e-2 (bf16), LSE 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gen import DECODE_WORKLOADS, make_qkv_kv

TOL_O = {"fp16": 4e-3, "bf16": 3.2e-2}
TOL_LSE = 1e-3
ALIGN = {"causal": "top_left", "causal_bottom_right": "bottom_right"}


def _oracle(q, k, v, mask, scale):
    if mask == "none":
        return oracle.attn_fwd_qk(q, k, v, False, scale)
    return oracle.attn_fwd_qk(q, k, v, True, scale, align=ALIGN[mask])


def _compare(name, o, lse, o_ref, lse_ref, dtype):
    o64 = o.to(torch.float64).cpu().numpy()
    l64 = lse.to(torch.float64).cpu().numpy()
    empty = np.isneginf(lse_ref)
    # rows with no visible key: exactly O = 0 and LSE = -inf
    assert np.array_equal(np.isneginf(l64), empty), f"{name}: -inf LSE rows differ"
    assert (o64[empty] == 0).all(), f"{name}: a row without keys has O != 0"
    assert np.isfinite(o64).all(), f"{name}: non-finite O"
    eo = np.abs(o64 - o_ref).max(initial=0.0)
    el = np.abs(l64[~empty] - lse_ref[~empty]).max(initial=0.0)
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, \
        f"{name}: max|dO| = {eo:.3e} (tol {TOL_O[dtype]}), max|dLSE| = {el:.3e} (tol {TOL_LSE})"
    return eo, el


def _case(attn, B, H, Nq, Nk, d, dtype, mask, seed, workspace=None, scale=None):
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, dtype, seed)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = attn.fwd_kv(q.cuda(), k.cuda(), v.cuda(), mask=mask, scale=scale,
                         workspace=workspace, checked=True)
    o_ref, lse_ref = _oracle(q, k, v, mask, scale)
    _compare(f"B{B}H{H}q{Nq}k{Nk}d{d}{dtype}-{mask}", o, lse, o_ref, lse_ref, dtype)
    return q, k, v, o, lse


@pytest.mark.gpu
@pytest.mark.parametrize("w", DECODE_WORKLOADS, ids=lambda w: w.name)
@pytest.mark.parametrize("mask", ["none", "causal_bottom_right"])
def test_decode_workloads(cuda_lib, w, mask):
    # every decode workload runs the streaming decode kernel over several key ranges
    assert cuda_lib.workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d) > 0
    _case(cuda_lib, w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, mask, w.seed)


@pytest.mark.gpu
@pytest.mark.parametrize("Nq", [1, 2, 3, 16, 64])
@pytest.mark.parametrize("Nk", [1, 127, 128, 129, 1000, 5000])
@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16")])
def test_decode_grid(cuda_lib, Nq, Nk, d, dtype):
    for mask in ("none", "causal", "causal_bottom_right"):
        _case(cuda_lib, 2, 3, Nq, Nk, d, dtype, mask, seed=Nq * 10007 + Nk * 7 + d)


@pytest.mark.gpu
@pytest.mark.parametrize("Nq,Nk", [(1000, 300), (300, 1000), (257, 129), (129, 4097), (513, 1),
                                   (600, 600)])
@pytest.mark.parametrize("mask", ["none", "causal", "causal_bottom_right"])
@pytest.mark.parametrize("split", [True, False])
def test_cross_lengths(cuda_lib, Nq, Nk, mask, split):
    _case(cuda_lib, 1, 4, Nq, Nk, 64, "bf16", mask, seed=Nq * 31 + Nk,
          workspace=None if split else False)


@pytest.mark.gpu
def test_rows_without_keys(cuda_lib):
    """Bottom-right alignment with Nq > Nk: the first Nq - Nk rows see no key. With
    Nq - Nk >= 256 whole CTAs (and with 128 whole Q tiles) see no key at all."""
    for Nq, Nk in ((700, 100), (300, 40), (130, 3)):
        _case(cuda_lib, 1, 2, Nq, Nk, 128, "fp16", "causal_bottom_right", seed=Nq + Nk)


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_square_matches_attn_fwd_bitwise(cuda_lib, mask):
    """Without a workspace, attn_fwd_kv with Nq = Nk runs the same kernel as attn_fwd."""
    q, k, v = (t.cuda() for t in make_qkv_kv(2, 4, 1000, 1000, 64, "bf16", seed=5))
    o1, l1 = cuda_lib.fwd(q, k, v, causal=mask == "causal", checked=True)
    o2, l2 = cuda_lib.fwd_kv(q, k, v, mask=mask, workspace=False, checked=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # bottom-right equals top-left when Nq = Nk
    o3, l3 = cuda_lib.fwd_kv(q, k, v, mask="causal_bottom_right" if mask == "causal" else "none",
                             workspace=False, checked=True)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


@pytest.mark.gpu
def test_split_matches_unsplit_and_is_deterministic(cuda_lib):
    q, k, v = (t.cuda() for t in make_qkv_kv(1, 8, 4, 30000, 128, "bf16", seed=9))
    n = cuda_lib.workspace_bytes(1, 8, 4, 30000, 128)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o1, l1 = cuda_lib.fwd_kv(q, k, v, mask="causal_bottom_right", workspace=ws, checked=True)
    o2, l2 = cuda_lib.fwd_kv(q, k, v, mask="causal_bottom_right", workspace=ws, checked=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = cuda_lib.fwd_kv(q, k, v, mask="causal_bottom_right", workspace=False, checked=True)
    assert (o1.float() - o3.float()).abs().max().item() <= 2 * TOL_O["bf16"] / 4
    assert (l1 - l3).abs().max().item() <= 1e-4
    # a smaller workspace gives fewer ranges: same result within rounding
    o4, l4 = cuda_lib.fwd_kv(q, k, v, mask="causal_bottom_right", workspace=ws[: n // 3 + 16],
                             checked=True)
    assert (o1.float() - o4.float()).abs().max().item() <= 2 * TOL_O["bf16"] / 4
    assert (l1 - l4).abs().max().item() <= 1e-4


@pytest.mark.gpu
def test_workspace_needs_no_initialisation(cuda_lib):
    q, k, v = (t.cuda() for t in make_qkv_kv(2, 2, 1, 3000, 64, "fp16", seed=11))
    n = cuda_lib.workspace_bytes(2, 2, 1, 3000, 64)
    ws_nan = torch.full((n // 4,), float("nan"), dtype=torch.float32, device="cuda").view(torch.uint8)
    ws_zero = torch.zeros(n, dtype=torch.uint8, device="cuda")
    o1, l1 = cuda_lib.fwd_kv(q, k, v, workspace=ws_nan, checked=True)
    o2, l2 = cuda_lib.fwd_kv(q, k, v, workspace=ws_zero, checked=True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
