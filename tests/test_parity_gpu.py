"""Parity of the CUDA forward (through the C ABI) with the fp64 CPU oracle.

Tolerances (max-abs, per element): O within 4e-3 for fp16 and 3.2e-2 for bf16;
LSE within 1e-3. Every element is compared for the small problems, for the headline
problem under both masks and for the x2-scaled long problem: the multithreaded C
oracle computes those in seconds. Those three also report their error budget (max
error, elements over tolerance, and the error against the oracle rounded to the
output dtype, i.e. what is left beside the final rounding). The 48 points of the
sequence sweep are compared on two rows of every 128-row tile of every head, plus
properties that hold at any size (causal row 0 equals V[0] exactly, outputs finite
and inside the range of V).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gen import make_qkv, make_qkv_rising, sweep_points, workload

TOL_O = {"fp16": 4e-3, "bf16": 3.2e-2}
TOL_LSE = 1e-3


def _run(attn, q, k, v, causal, scale):
    o, lse = attn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, checked=True)
    return o.cpu(), lse.cpu()


def _report(name, o_gpu, lse_gpu, o_ref, lse_ref, dtype):
    o64 = o_gpu.to(torch.float64).numpy().reshape(o_ref.shape)
    l64 = lse_gpu.to(torch.float64).numpy().reshape(lse_ref.shape)
    assert np.isfinite(o64).all() and np.isfinite(l64).all(), f"{name}: non-finite output"
    eo = np.abs(o64 - o_ref)
    el = np.abs(l64 - lse_ref)
    tol = TOL_O[dtype]
    msg = (f"{name}: max|dO| = {eo.max():.3e} (tol {tol}, {int((eo > tol).sum())} over), "
           f"max|dLSE| = {el.max():.3e} (tol {TOL_LSE}, {int((el > TOL_LSE).sum())} over)")
    assert eo.max() <= tol and el.max() <= TOL_LSE, msg
    return eo.max(), el.max()


def _full(attn, B, H, N, d, dtype, causal, seed, input_scale=1.0):
    q, k, v = make_qkv(B, H, N, d, dtype, seed, input_scale)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(attn, q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    return _report(f"B{B}H{H}N{N}d{d}{dtype}{'c' if causal else ''}", o, lse, o_ref, lse_ref, dtype)


def _sample_rows(BH, N, rng):
    """Two rows of every 128-row tile of every head: one at a random offset inside the
    tile and its first or last row (alternating), plus the last row of the sequence."""
    rows = []
    for h in range(BH):
        for t0 in range(0, N, 128):
            n = min(128, N - t0)
            r = {t0 + int(rng.integers(0, n)), t0 if (t0 // 128) % 2 == 0 else t0 + n - 1}
            rows.extend(h * N + x for x in sorted(r))
        rows.append(h * N + N - 1)
    return np.unique(np.array(rows, dtype=np.int64))


def _sampled(attn, B, H, N, d, dtype, causal, seed, input_scale=1.0):
    q, k, v = make_qkv(B, H, N, d, dtype, seed, input_scale)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(attn, q, k, v, causal, scale)
    rows = _sample_rows(B * H, N, np.random.default_rng(seed))
    o_ref, lse_ref = oracle.attn_fwd_rows(q, k, v, causal, rows, scale)
    og = o.reshape(-1, d)[torch.from_numpy(rows)]
    lg = lse.reshape(-1)[torch.from_numpy(rows)]
    name = f"B{B}H{H}N{N}d{d}{dtype}{'c' if causal else ''}x{input_scale:g}"
    _report(name, og, lg, o_ref, lse_ref, dtype)
    # properties over every output
    of = o.to(torch.float32)
    assert torch.isfinite(of).all() and torch.isfinite(lse).all(), f"{name}: non-finite"
    vf = v.to(torch.float32)
    vmax = vf.amax(dim=2, keepdim=True)
    vmin = vf.amin(dim=2, keepdim=True)
    tol = TOL_O[dtype]
    assert (of <= vmax + tol).all() and (of >= vmin - tol).all(), f"{name}: O outside range of V"
    if causal:
        assert torch.equal(o[:, :, 0], v[:, :, 0]), f"{name}: causal row 0 differs from V[0]"
    return o, lse


def _whole(attn, B, H, N, d, dtype, causal, seed, input_scale=1.0):
    """Every element against the oracle, with the error budget reported."""
    import json
    import os
    q, k, v = make_qkv(B, H, N, d, dtype, seed, input_scale)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(attn, q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    name = f"B{B}H{H}N{N}d{d}{dtype}{'c' if causal else ''}x{input_scale:g}"
    o64 = o.to(torch.float64).numpy()
    # the oracle rounded once to the output dtype: the part of the error that is not
    # the output's own rounding
    o_ref_rounded = torch.from_numpy(o_ref).to(o.dtype).to(torch.float64).numpy()
    tol = TOL_O[dtype]
    eo = np.abs(o64 - o_ref)
    el = np.abs(lse.to(torch.float64).numpy() - lse_ref)
    rep = {"problem": name, "elements": int(eo.size), "max_abs_dO": float(eo.max()),
           "over_tol_O": int((eo > tol).sum()), "tol_O": tol,
           "max_abs_dO_vs_rounded_oracle": float(np.abs(o64 - o_ref_rounded).max()),
           "max_abs_dLSE": float(el.max()), "over_tol_LSE": int((el > TOL_LSE).sum()), "tol_LSE": TOL_LSE}
    print("PARITY_REPORT " + json.dumps(rep))
    path = os.environ.get("ATTN_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rep) + "\n")
    _report(name, o, lse, o_ref, lse_ref, dtype)
    if causal:
        assert torch.equal(o[:, :, 0], v[:, :, 0]), f"{name}: causal row 0 differs from V[0]"
    return rep


# ---- the named workloads ------------------------------------------------------------------

@pytest.mark.gpu
def test_smallest(cuda_lib):
    w = workload("b1h1n128d64")
    _full(cuda_lib, w.B, w.H, w.N, w.d, "fp16", False, w.seed)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_boundary_n1000(cuda_lib, dtype, causal):
    w = workload("b2h4n1000d64")
    _full(cuda_lib, w.B, w.H, w.N, w.d, dtype, causal, w.seed)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_headline_b4h16n4096d64(cuda_lib, causal):
    w = workload("b4h16n4096d64")
    _whole(cuda_lib, w.B, w.H, w.N, w.d, "bf16", causal, w.seed)


@pytest.mark.gpu
def test_long_b1h16n8192d128_scaled(cuda_lib):
    w = workload("b1h16n8192d128x2")
    _whole(cuda_lib, w.B, w.H, w.N, w.d, "bf16", True, w.seed, w.input_scale)


@pytest.mark.gpu
@pytest.mark.parametrize("pt", list(sweep_points()),
                         ids=lambda p: f"N{p['N']}d{p['d']}{p['dtype']}{'c' if p['causal'] else ''}")
def test_sweep(cuda_lib, pt):
    _sampled(cuda_lib, pt["B"], pt["H"], pt["N"], pt["d"], pt["dtype"], pt["causal"], pt["seed"])


# ---- edge shapes: ragged tails, single key, one tile, tile +- 1 ------------------------------

EDGE_N = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 384, 513]


@pytest.mark.gpu
@pytest.mark.parametrize("N", EDGE_N)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_shapes(cuda_lib, N, d, dtype, causal):
    _full(cuda_lib, 1, 3, N, d, dtype, causal, seed=9000 + N * 4 + d)


@pytest.mark.gpu
def test_nondefault_scale_and_many_heads(cuda_lib):
    q, k, v = make_qkv(3, 5, 300, 64, "bf16", seed=4242)
    for causal in (False, True):
        o, lse = _run(cuda_lib, q, k, v, causal, 0.37)
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 0.37)
        _report("scale0.37", o, lse, o_ref, lse_ref, "bf16")


@pytest.mark.gpu
def test_deterministic_and_unchecked_path(cuda_lib):
    q, k, v = (t.cuda() for t in make_qkv(2, 4, 1000, 64, "bf16", seed=11))
    for causal in (False, True):
        o1, l1 = cuda_lib.fwd(q, k, v, causal=causal, checked=True)
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            o2, l2 = cuda_lib.fwd(q, k, v, causal=causal)
        stream.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert cuda_lib.device_error_info() == [0, 0, 0, 0]


@pytest.mark.gpu
def test_rejects_bad_device_arguments(cuda_lib):
    from exact_attention_61_gb300.attn import AttnError
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 64, 96, "bf16", seed=1))
    with pytest.raises(AttnError) as e:
        cuda_lib.fwd(q, k, v)
    assert e.value.status == 2
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 64, 64, "bf16", seed=1))
    with pytest.raises(AttnError):
        cuda_lib.fwd(q, k, v, scale=-1.0)


# ---- online rescaling on every tile ------------------------------------------------------------

@pytest.mark.gpu
@pytest.mark.parametrize("N", [200, 384, 513, 1000, 2048])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_rising_scores_rescale_every_tile(cuda_lib, N, d, dtype, causal):
    """Scores rise along the keys, so each key tile raises the row maximum by more than
    the lazy-rescale threshold: O is rescaled in TMEM on every tile. N=384 and N=513
    leave the last CTA with a single Q tile."""
    q, k, v = make_qkv_rising(1, 2, N, d, dtype, seed=7000 + N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = _run(cuda_lib, q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    _report(f"rising N{N}d{d}{dtype}{'c' if causal else ''}", o, lse, o_ref, lse_ref, dtype)
