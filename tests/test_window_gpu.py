"""Parity of the sliding-window / key-padding forward (attn_fwd_window, through the
C ABI) with the fp64 oracle (oracle.attn_fwd_window): windows of many widths in both
alignments, causal and two-sided, per-batch key counts including empty sequences
(rows with no visible key must be exactly O = 0, LSE = -inf), windows that leave
whole CTAs and Q tiles without keys, and the split of the keys for decoding.

Tolerances as for the other forwards: O max-abs 4e-3 (fp16) / 3.2e-2 (bf16), LSE 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gen import make_qkv_kv

TOL_O = {"fp16": 4e-3, "bf16": 3.2e-2}
TOL_LSE = 1e-3


def _case(attn, B, H, Nq, Nk, d, dtype, window, lens, align, seed, workspace=None):
    q, k, v = make_qkv_kv(B, H, Nq, Nk, d, dtype, seed)
    scale = 1.0 / math.sqrt(d)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    o, lse = attn.fwd_window(q.cuda(), k.cuda(), v.cuda(), window=window, kv_lens=kl, align=align,
                             scale=scale, workspace=workspace, checked=True)
    o_ref, lse_ref = oracle.attn_fwd_window(q, k, v, window[0], window[1], lens, align, scale)
    name = f"B{B}H{H}q{Nq}k{Nk}d{d}{dtype} w{window} lens{lens} {align}"
    o64 = o.double().cpu().numpy()
    l64 = lse.double().cpu().numpy()
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l64), empty), f"{name}: rows without keys differ"
    assert (o64[empty] == 0).all(), f"{name}: a row without keys has O != 0"
    assert np.isfinite(o64).all(), f"{name}: non-finite O"
    eo = np.abs(o64 - o_ref).max(initial=0.0)
    el = np.abs(l64[~empty] - lse_ref[~empty]).max(initial=0.0)
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, f"{name}: max|dO| {eo:.3e}, max|dLSE| {el:.3e}"


WINDOWS = [(0, 0), (1, 0), (63, 0), (127, 0), (128, 0), (200, 0), (255, 0), (256, 0), (511, 0),
           (64, 64), (100, 300), (-1, 5), (300, -1), (-1, 0), (-1, -1)]


@pytest.mark.gpu
@pytest.mark.parametrize("window", WINDOWS, ids=str)
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "fp16")])
def test_square_windows(cuda_lib, window, d, dtype):
    _case(cuda_lib, 2, 3, 1000, 1000, d, dtype, window, None, "top_left",
          seed=63000 + 7 * window[0] + window[1] + d)


@pytest.mark.gpu
@pytest.mark.parametrize("lens", [[1000, 999, 513, 256, 255, 129, 1, 0]], ids=["mixed"])
@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (100, 0), (0, 0)], ids=str)
@pytest.mark.parametrize("align", ["top_left", "bottom_right"])
def test_padding(cuda_lib, lens, window, align):
    _case(cuda_lib, 8, 2, 700, 1000, 64, "bf16", window, lens, align, seed=63100 + window[0] % 7)


@pytest.mark.gpu
@pytest.mark.parametrize("Nq,Nk", [(1, 5000), (4, 9000), (16, 1000), (300, 1000), (1000, 300)])
@pytest.mark.parametrize("window", [(1024, 0), (4095, 0), (50, 10), (-1, 0)], ids=str)
@pytest.mark.parametrize("split", [True, False])
def test_decode_windows(cuda_lib, Nq, Nk, window, split):
    lens = [Nk, max(1, Nk // 3)]
    _case(cuda_lib, 2, 4, Nq, Nk, 128, "bf16", window, lens, "bottom_right", seed=63200 + Nq + Nk,
          workspace=None if split else False)


@pytest.mark.gpu
def test_no_window_matches_attn_fwd_bitwise(cuda_lib):
    q, k, v = (t.cuda() for t in make_qkv_kv(2, 4, 1000, 1000, 64, "bf16", 63300))
    for causal in (False, True):
        o1, l1 = cuda_lib.fwd(q, k, v, causal=causal, checked=True)
        o2, l2 = cuda_lib.fwd_window(q, k, v, window=(-1, 0 if causal else -1), workspace=False, checked=True)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
