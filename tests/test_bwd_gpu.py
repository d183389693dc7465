"""Parity of the CUDA backward (attn_bwd through the C ABI) with the fp64 oracle.

Tolerance, per element, derived from the arithmetic of the path (the pages state
none for the backward); the bound and its derivation are in oracle/bwd_bound.py:
P, dS and the outputs rounded to the dtype, fp32 sums, and D = dO . O formed from the
16-bit O. Every element must be within twice its bound (plus 1e-6 absolute for exact
zeros).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gen import make_qkv
from oracle import bwd_bound

U = bwd_bound.U
DT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _inputs(B, H, N, d, dtype, seed, scale_in=1.0):
    q, k, v = make_qkv(B, H, N, d, dtype, seed, scale_in)
    do = make_qkv(B, H, N, d, dtype, seed + 7919)[0]
    return q, k, v, do


_d_error = bwd_bound.d_error


def _check(name, got, ref, m, q64, k64, do64, dD, scale, dtype, N):
    bnd = bwd_bound.bounds(ref, m, q64, k64, do64, dD, scale, dtype, N)
    ok, msg = bwd_bound.check({key: t.to(torch.float64).cpu().numpy() for key, t in got.items()}, ref, bnd)
    assert ok, f"{name}: {msg}"


def _run(attn, q, k, v, do, o, lse, causal, scale):
    dq, dk, dv = attn.bwd(q, k, v, o, lse, do, causal=causal, scale=scale, checked=True)
    return {"dq": dq, "dk": dk, "dv": dv}


def _case(attn, B, H, N, d, dtype, causal, seed, e2e=False, scale=None, scale_in=1.0):
    q, k, v, do = _inputs(B, H, N, d, dtype, seed, scale_in)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q64, k64, v64, do64 = (oracle.to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    gq, gk, gv, gdo = (t.cuda() for t in (q, k, v, do))
    if e2e:  # O and LSE from the CUDA forward
        o, lse = attn.fwd(gq, gk, gv, causal=causal, scale=scale, checked=True)
    else:    # O and LSE from the oracle, rounded as the forward's outputs are
        o = torch.from_numpy(o_ref).to(DT[dtype]).cuda()
        lse = torch.from_numpy(lse_ref).to(torch.float32).cuda()
    got = _run(attn, gq, gk, gv, gdo, o, lse, causal, scale)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, scale)
    m = oracle.attn_bwd_materialised(q, k, v, do, causal, scale)
    dD = _d_error(do64, o.to(torch.float64).cpu().numpy(), o_ref, U[dtype])
    name = f"B{B}H{H}N{N}d{d}{dtype}{'c' if causal else ''}{'-e2e' if e2e else ''}"
    _check(name, got, {"dq": dq, "dk": dk, "dv": dv}, m, q64, k64, do64, dD, scale, dtype, N)
    return got


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_boundary_n1000(cuda_lib, dtype, causal):
    _case(cuda_lib, 2, 4, 1000, 64, dtype, causal, seed=62001)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_smallest(cuda_lib, causal):
    _case(cuda_lib, 1, 1, 128, 64, "fp16", causal, seed=62000)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [1, 2, 63, 127, 128, 129, 255, 256, 257, 384, 513])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_edge_shapes(cuda_lib, N, d, dtype):
    for causal in (False, True):
        _case(cuda_lib, 1, 3, N, d, dtype, causal, seed=62100 + N * 4 + d + len(dtype))


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_end_to_end_with_cuda_forward(cuda_lib, d, causal):
    _case(cuda_lib, 2, 2, 777, d, "bf16", causal, seed=62200 + d, e2e=True)


@pytest.mark.gpu
def test_scaled_inputs_and_scale(cuda_lib):
    _case(cuda_lib, 1, 4, 640, 128, "bf16", True, seed=62300, scale=0.37, scale_in=2.0)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_headline_size_sampled_heads(cuda_lib, causal):
    """B=4, H=16, N=4096, d=64, bf16: the whole problem runs on the GPU; three heads
    are checked element by element against the oracle on those heads alone."""
    B, H, N, d, dtype = 4, 16, 4096, 64, "bf16"
    q, k, v, do = _inputs(B, H, N, d, dtype, seed=62400 + int(causal))
    scale = 1.0 / math.sqrt(d)
    gq, gk, gv, gdo = (t.cuda() for t in (q, k, v, do))
    o, lse = cuda_lib.fwd(gq, gk, gv, causal=causal, scale=scale, checked=True)
    got = _run(cuda_lib, gq, gk, gv, gdo, o, lse, causal, scale)
    for b, h in ((0, 0), (1, 7), (3, 15)):
        sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
        qs, ks, vs, dos = (sl(t) for t in (q, k, v, do))
        o_ref, _ = oracle.attn_fwd(qs, ks, vs, causal, scale)
        dq, dk, dv = oracle.attn_bwd(qs, ks, vs, dos, causal, scale)
        m = oracle.attn_bwd_materialised(qs, ks, vs, dos, causal, scale)
        dD = _d_error(oracle.to_f64(dos), sl(o).to(torch.float64).cpu().numpy(), o_ref, U[dtype])
        g = {key: sl(t) for key, t in got.items()}
        _check(f"headline b{b}h{h}{'c' if causal else ''}", g, {"dq": dq, "dk": dk, "dv": dv}, m,
               oracle.to_f64(qs), oracle.to_f64(ks), oracle.to_f64(dos), dD, scale, dtype, N)
        del m


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_d128_large_sampled_heads(cuda_lib, causal):
    """B=2, H=8, N=3000 (ragged), d=128, fp16: the whole problem on the GPU, two heads
    checked element by element (the d=128 dQ path stages in the Q/dO ring)."""
    B, H, N, d, dtype = 2, 8, 3000, 128, "fp16"
    q, k, v, do = _inputs(B, H, N, d, dtype, seed=62700 + int(causal))
    scale = 1.0 / math.sqrt(d)
    gq, gk, gv, gdo = (t.cuda() for t in (q, k, v, do))
    o, lse = cuda_lib.fwd(gq, gk, gv, causal=causal, scale=scale, checked=True)
    got = _run(cuda_lib, gq, gk, gv, gdo, o, lse, causal, scale)
    for b, h in ((0, 3), (1, 7)):
        sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
        qs, ks, vs, dos = (sl(t) for t in (q, k, v, do))
        o_ref, _ = oracle.attn_fwd(qs, ks, vs, causal, scale)
        dq, dk, dv = oracle.attn_bwd(qs, ks, vs, dos, causal, scale)
        m = oracle.attn_bwd_materialised(qs, ks, vs, dos, causal, scale)
        dD = _d_error(oracle.to_f64(dos), sl(o).to(torch.float64).cpu().numpy(), o_ref, U[dtype])
        g = {key: sl(t) for key, t in got.items()}
        _check(f"d128 b{b}h{h}{'c' if causal else ''}", g, {"dq": dq, "dk": dk, "dv": dv}, m,
               oracle.to_f64(qs), oracle.to_f64(ks), oracle.to_f64(dos), dD, scale, dtype, N)
        del m


@pytest.mark.gpu
def test_dk_dv_deterministic_and_dq_reproducible(cuda_lib):
    q, k, v, do = (t.cuda() for t in _inputs(2, 4, 1500, 64, "bf16", seed=62500))
    o, lse = cuda_lib.fwd(q, k, v, causal=True, checked=True)
    a = cuda_lib.bwd(q, k, v, o, lse, do, causal=True, checked=True)
    b = cuda_lib.bwd(q, k, v, o, lse, do, causal=True, checked=True)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    # dQ sums key tiles with fp32 atomics: the order may differ, the value barely
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2 * 2.0 ** -8 * a[0].float().abs().max().item()


@pytest.mark.gpu
def test_sum_rules_hold_on_the_gpu(cuda_lib):
    """sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i (softmax rows sum to one), at a
    size the oracle would need long for: B=1, H=8, N=8192, d=128, bf16, causal."""
    q, k, v, do = (t.cuda() for t in _inputs(1, 8, 8192, 128, "bf16", seed=62600))
    o, lse = cuda_lib.fwd(q, k, v, causal=True, checked=True)
    dq, dk, dv = cuda_lib.bwd(q, k, v, o, lse, do, causal=True, checked=True)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    dks = dk.double().sum(dim=2)
    scale_k = (dk.double().abs().sum(dim=2)).clamp_min(1e-30)
    assert (dks.abs() / scale_k).max().item() < 3e-2
    dvs = dv.double().sum(dim=2)
    dos = do.double().sum(dim=2)
    assert ((dvs - dos).abs() / dv.double().abs().sum(dim=2)).max().item() < 3e-2


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_headline_size_every_head_identities(cuda_lib, causal):
    """B=4, H=16, N=4096, d=64, bf16 (the persistent d=64 backward: 2048 key-tile items over
    the SMs; causal items claimed from a counter). Every head satisfies
    sum_j dK_j = 0, sum_j dV_j = sum_i dO_i, and sum_i q_i . dQ_i = sum_j k_j . dK_j (scaling
    Q or K scales the scores alike). The last ties dQ, summed over every key-tile item of
    the head, to dK: an item whose dQ is lost or added twice breaks it."""
    B, H, N, d = 4, 16, 4096, 64
    q, k, v, do = (t.cuda() for t in _inputs(B, H, N, d, "bf16", seed=62800 + int(causal)))
    o, lse = cuda_lib.fwd(q, k, v, causal=causal, checked=True)
    dq, dk, dv = cuda_lib.bwd(q, k, v, o, lse, do, causal=causal, checked=True)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    dk64, dv64, dq64 = dk.double(), dv.double(), dq.double()
    rel = lambda a, b, s: ((a - b).abs() / s.clamp_min(1e-30)).max().item()
    assert rel(dk64.sum(dim=2), 0.0, dk64.abs().sum(dim=2)) < 3e-2
    assert rel(dv64.sum(dim=2), do.double().sum(dim=2), dv64.abs().sum(dim=2)) < 3e-2
    qdq = q.double() * dq64
    kdk = k.double() * dk64
    assert rel(qdq.sum(dim=(2, 3)), kdk.sum(dim=(2, 3)), qdq.abs().sum(dim=(2, 3)) + kdk.abs().sum(dim=(2, 3))) < 5e-3
