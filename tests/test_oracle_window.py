"""Pins of the sliding-window / key-padding oracle (oracle.attn_fwd_window): reductions
to the pinned Nq-against-Nk oracle (no window, causal in both alignments, padding as
slicing), closed forms (a one-key window gives V of the diagonal key exactly; an empty
padded sequence gives O = 0 and LSE = -inf), and brute force on tiny inputs with the
visible set enumerated in plain Python and the arithmetic done by torch SDPA."""
import math

import numpy as np
import pytest
import torch

import oracle

TIGHT = 1e-12


def _rand(B, H, Nq, Nk, d, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((B, H, Nq, d)), g.standard_normal((B, H, Nk, d)), g.standard_normal((B, H, Nk, d))


@pytest.mark.parametrize("Nq,Nk", [(5, 5), (3, 17), (20, 6), (64, 64)])
def test_reduces_to_qk_oracle(Nq, Nk):
    q, k, v = _rand(2, 2, Nq, Nk, 8, seed=Nq * 100 + Nk)
    o, l = oracle.attn_fwd_window(q, k, v, -1, -1, scale=0.4)
    o2, l2 = oracle.attn_fwd_qk(q, k, v, False, 0.4)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(l, l2)
    for align in ("top_left", "bottom_right"):
        o, l = oracle.attn_fwd_window(q, k, v, -1, 0, align=align, scale=0.4)
        o2, l2 = oracle.attn_fwd_qk(q, k, v, True, 0.4, align=align)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(l, l2)
    # a window wider than the keys on both sides is no window at all
    o, l = oracle.attn_fwd_window(q, k, v, Nk + Nq, Nk + Nq, scale=0.4)
    o2, l2 = oracle.attn_fwd_qk(q, k, v, False, 0.4)
    np.testing.assert_allclose(o, o2, atol=TIGHT)


def test_one_key_window_is_that_key():
    q, k, v = _rand(1, 3, 9, 9, 4, seed=3)
    o, l = oracle.attn_fwd_window(q, k, v, 0, 0, scale=0.7)
    np.testing.assert_array_equal(o, v)
    np.testing.assert_allclose(l, 0.7 * (q * k).sum(-1), atol=TIGHT)
    # bottom-right with fewer queries: row i's only key is i + Nk - Nq
    q2 = q[:, :, :4]
    o, _ = oracle.attn_fwd_window(q2, k, v, 0, 0, align="bottom_right", scale=0.7)
    np.testing.assert_array_equal(o, v[:, :, 5:])


def test_padding_is_slicing_and_empty_rows():
    B, H, Nq, Nk, d = 3, 2, 6, 40, 8
    q, k, v = _rand(B, H, Nq, Nk, d, seed=5)
    lens = [40, 17, 0]
    for align in ("top_left", "bottom_right"):
        for causal in (False, True):
            o, l = oracle.attn_fwd_window(q, k, v, -1, 0 if causal else -1, lens, align, scale=0.3)
            for b, n in enumerate(lens):
                if n == 0:
                    assert np.all(o[b] == 0) and np.all(np.isneginf(l[b]))
                    continue
                ob, lb = oracle.attn_fwd_qk(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n], causal, 0.3,
                                            align=align)
                np.testing.assert_array_equal(o[b:b + 1], ob)
                np.testing.assert_array_equal(l[b:b + 1], lb)


@pytest.mark.parametrize("left,right", [(2, 0), (0, 3), (3, 1), (5, -1), (-1, 2), (1, 1)])
@pytest.mark.parametrize("align", ["top_left", "bottom_right"])
def test_brute_force_visible_sets(left, right, align):
    B, H, Nq, Nk, d = 2, 1, 7, 11, 5
    q, k, v = _rand(B, H, Nq, Nk, d, seed=left * 10 + right + 50)
    lens = [11, 8]
    o, l = oracle.attn_fwd_window(q, k, v, left, right, lens, align, scale=0.9)
    for b in range(B):
        n = lens[b]
        for i in range(Nq):
            diag = i + (n - Nq if align == "bottom_right" else 0)
            vis = [j for j in range(n)
                   if (left < 0 or j >= diag - left) and (right < 0 or j <= diag + right)]
            if not vis:
                assert np.all(o[b, 0, i] == 0) and np.isneginf(l[b, 0, i])
                continue
            qi = torch.tensor(q[b, 0, i:i + 1])
            kv_k = torch.tensor(k[b, 0, vis])
            kv_v = torch.tensor(v[b, 0, vis])
            ref = torch.nn.functional.scaled_dot_product_attention(qi[None], kv_k[None], kv_v[None], scale=0.9)
            np.testing.assert_allclose(o[b, 0, i], ref[0, 0].numpy(), atol=TIGHT)
            s = 0.9 * (kv_k @ qi[0])
            assert abs(l[b, 0, i] - torch.logsumexp(s, 0).item()) < TIGHT


def test_window_mask_helper_matches_the_oracle():
    """The boolean helper the GPU tests use agrees with the oracle's visible sets."""
    B, H, Nq, Nk, d = 2, 1, 9, 13, 4
    q, k, v = _rand(B, H, Nq, Nk, d, seed=77)
    for left, right, lens, align in [(3, 0, [13, 5], "top_left"), (2, 2, [10, 13], "bottom_right"),
                                     (-1, 0, None, "bottom_right")]:
        o, l = oracle.attn_fwd_window(q, k, v, left, right, lens, align, scale=0.5)
        keep = oracle.window_mask(B, Nq, Nk, left, right, lens, align)
        s = 0.5 * np.einsum("bhid,bhjd->bhij", q, k)
        s = np.where(keep[:, None], s, -np.inf)
        m = np.max(s, axis=-1, keepdims=True)
        e = np.where(np.isfinite(m), np.exp(s - np.where(np.isfinite(m), m, 0)), 0)
        ref = np.einsum("bhij,bhjd->bhid", e, v) / np.maximum(e.sum(-1, keepdims=True), 1e-300)
        np.testing.assert_allclose(o, ref, atol=TIGHT)
