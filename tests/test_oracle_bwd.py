"""Pins of the fp64 backward oracle (oracle.attn_bwd) to things other than itself:
torch float64 autograd through an explicit forward, central finite differences of
the pinned forward oracle, closed forms (one key, causal row 0, the last key under
the causal mask), sum rules (sum_j dK_j = 0, sum_j dV_j = sum_i dO_i), and planted
mistakes that each of these catches."""
import numpy as np
import pytest
import torch

import oracle
from gen import make_qkv

TIGHT = 1e-11


def _rand(B, H, N, d, seed, n=4):
    g = np.random.default_rng(seed)
    return [g.standard_normal((B, H, N, d)) for _ in range(n)]


def _torch_grads(q, k, v, do, causal, scale):
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * q @ k.transpose(-1, -2)
    if causal:
        N = s.shape[-1]
        s = s.masked_fill(~torch.ones(N, N, dtype=torch.bool).tril(), float("-inf"))
    o = torch.softmax(s, dim=-1) @ v
    (o * torch.tensor(do)).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("N,d", [(1, 4), (2, 3), (7, 5), (64, 16), (130, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_autograd(N, d, causal):
    q, k, v, do = _rand(2, 2, N, d, seed=N * 13 + d)
    scale = 0.7 / np.sqrt(d)
    got = oracle.attn_bwd(q, k, v, do, causal, scale)
    want = _torch_grads(q, k, v, do, causal, scale)
    for g, w, name in zip(got, want, ("dq", "dk", "dv")):
        np.testing.assert_allclose(g, w, rtol=0, atol=TIGHT * max(1.0, np.abs(w).max()), err_msg=name)


@pytest.mark.parametrize("causal", [False, True])
def test_materialised_twin_agrees(causal):
    q, k, v, do = _rand(1, 3, 50, 8, seed=5)
    got = oracle.attn_bwd(q, k, v, do, causal, 0.3)
    m = oracle.attn_bwd_materialised(q, k, v, do, causal, 0.3)
    for g, name in zip(got, ("dq", "dk", "dv")):
        np.testing.assert_allclose(g, m[name], rtol=0, atol=TIGHT)
    # D = rowsum(P * dP) equals dO . O, the form the FA2 backward uses
    o, _ = oracle.attn_fwd(q, k, v, causal, 0.3)
    np.testing.assert_allclose(m["D"], (do * o).sum(-1), rtol=0, atol=TIGHT)


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_of_the_forward_oracle(causal):
    """Central differences of L = sum(dO * O) with O from the (separately pinned)
    forward oracle, on a tiny problem, for every entry of Q, K and V."""
    q, k, v, do = _rand(1, 1, 5, 3, seed=11)
    scale, h = 0.9, 1e-5
    grads = oracle.attn_bwd(q, k, v, do, causal, scale)

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd(q_, k_, v_, causal, scale)
        return float((o * do).sum())

    for which, g in enumerate(grads):
        x = [q, k, v]
        for idx in np.ndindex(q.shape):
            plus = [a.copy() for a in x]
            minus = [a.copy() for a in x]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(fd - g[idx]) < 1e-8, (which, idx, fd, g[idx])


def test_closed_forms():
    # one key: O = V regardless of Q and K, so dQ = dK = 0 and dV = dO
    q, k, v, do = _rand(1, 2, 1, 6, seed=3)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, False, 0.5)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_array_equal(dv, do)
    # causal: row 0 sees one key, so its dQ is exactly zero; the last key is seen by
    # the last row only, so dV[N-1] = P[N-1, N-1] dO[N-1]
    q, k, v, do = _rand(1, 1, 9, 4, seed=4)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, True, 0.5)
    assert np.all(dq[0, 0, 0] == 0)
    s = 0.5 * q[0, 0, -1] @ k[0, 0].T
    p_last = np.exp(s[-1] - np.log(np.exp(s).sum()))
    np.testing.assert_allclose(dv[0, 0, -1], p_last * do[0, 0, -1], rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_sum_rules(causal):
    """Softmax rows sum to one: sum_j dS_ij = 0, hence sum_j dK_j = 0, and
    sum_j dV_j = sum_i dO_i."""
    q, k, v, do = _rand(2, 2, 77, 16, seed=6)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal, 0.25)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-11)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-11)


def test_sixteen_bit_inputs_match_torch():
    q, k, v = make_qkv(1, 2, 96, 64, "bf16", seed=12)
    do = make_qkv(1, 2, 96, 64, "bf16", seed=13)[0]
    got = oracle.attn_bwd(q, k, v, do, True, 0.125)
    want = _torch_grads(*(t.double().numpy() for t in (q, k, v, do)), True, 0.125)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, rtol=0, atol=1e-11)


# ---- planted mistakes: each plausible slip fails at least one pin above ------------------

def _mutant(q, k, v, do, causal, scale, kind):
    m = oracle.attn_bwd_materialised(q, k, v, do, causal, scale)
    p, dp, D = m["p"], m["dp"], m["D"][..., None]
    if kind == "D_sign":
        ds = p * (dp + D)
    elif kind == "no_D":
        ds = p * dp
    elif kind == "ds_transposed":
        ds = np.swapaxes(p * (dp - D), -1, -2)
    else:
        ds = p * (dp - D)
    sc_k = 1.0 if kind == "dk_no_scale" else scale
    dq = scale * np.einsum("bhij,bhjd->bhid", ds, k)
    dk = sc_k * np.einsum("bhij,bhid->bhjd", ds, q)
    pv = np.swapaxes(p, -1, -2) if kind == "dv_p_transposed" else p
    dv = np.einsum("bhij,bhid->bhjd", pv, do)
    return dq, dk, dv


@pytest.mark.parametrize("kind", ["D_sign", "no_D", "ds_transposed", "dk_no_scale",
                                  "dv_p_transposed"])
def test_planted_mistakes_are_caught(kind):
    q, k, v, do = _rand(1, 2, 12, 4, seed=21)
    causal, scale = True, 0.6
    good = _mutant(q, k, v, do, causal, scale, "none")
    for g, w in zip(good, _torch_grads(q, k, v, do, causal, scale)):
        np.testing.assert_allclose(g, w, atol=1e-12)
    bad = _mutant(q, k, v, do, causal, scale, kind)
    want = _torch_grads(q, k, v, do, causal, scale)
    caught_autograd = any(np.abs(b - w).max() > 1e-6 for b, w in zip(bad, want))
    caught_sums = (np.abs(bad[1].sum(axis=2)).max() > 1e-6 or
                   np.abs(bad[2].sum(axis=2) - do.sum(axis=2)).max() > 1e-6)
    assert caught_autograd
    if kind in ("D_sign", "no_D"):  # the sum rule alone catches a wrong D term
        assert caught_sums


# ---- windows, padding and Nq != Nk ------------------------------------------------------

def _torch_grads_mask(q, k, v, do, keep, scale):
    """torch float64 autograd through an explicit forward with a boolean [B,1|H,Nq,Nk]
    mask; rows without keys are given O = 0 (no gradient) as the oracle defines."""
    q, k, v = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    s = scale * q @ k.transpose(-1, -2)
    keep_t = torch.tensor(keep)
    s = s.masked_fill(~keep_t, float("-inf"))
    any_key = keep_t.any(-1, keepdim=True)
    p = torch.softmax(torch.where(any_key, s, torch.zeros_like(s)), dim=-1) * any_key
    o = p @ v
    (o * torch.tensor(do)).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("Nq,Nk,left,right,lens,align", [
    (9, 9, -1, -1, None, "top_left"),
    (9, 9, 3, 0, None, "top_left"),
    (5, 17, 4, 0, [17, 9], "bottom_right"),
    (12, 7, -1, 0, [7, 3], "bottom_right"),
    (8, 20, 2, 2, [20, 0], "top_left"),
    (6, 6, 0, 0, None, "top_left"),
])
def test_window_backward_matches_torch_autograd(Nq, Nk, left, right, lens, align):
    B, H, d = 2, 2, 4
    g = np.random.default_rng(Nq * 100 + Nk + left)
    q, do = g.standard_normal((B, H, Nq, d)), g.standard_normal((B, H, Nq, d))
    k, v = g.standard_normal((B, H, Nk, d)), g.standard_normal((B, H, Nk, d))
    got = oracle.attn_bwd_window(q, k, v, do, left, right, lens, align, scale=0.6)
    keep = oracle.window_mask(B, Nq, Nk, left, right, lens, align)[:, None]
    want = _torch_grads_mask(q, k, v, do, keep, 0.6)
    for a, w, name in zip(got, want, ("dq", "dk", "dv")):
        np.testing.assert_allclose(a, w, rtol=0, atol=1e-11, err_msg=name)
    if lens is not None:  # padded keys receive no gradient
        for b, n in enumerate(lens):
            assert np.all(got[1][b, :, n:] == 0) and np.all(got[2][b, :, n:] == 0)


def test_window_backward_reduces_to_square_and_finite_differences():
    q, k, v, do = _rand(1, 2, 10, 3, seed=31)
    for causal in (False, True):
        a = oracle.attn_bwd_window(q, k, v, do, -1, 0 if causal else -1, scale=0.8)
        b = oracle.attn_bwd(q, k, v, do, causal, 0.8)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
    # a two-sided window on a tiny problem: central differences of the windowed forward
    q, k, v, do = _rand(1, 1, 5, 3, seed=32)
    grads = oracle.attn_bwd_window(q, k, v, do, 1, 1, scale=0.9)

    def loss(q_, k_, v_):
        o, _ = oracle.attn_fwd_window(q_, k_, v_, 1, 1, scale=0.9)
        return float((o * do).sum())

    h = 1e-5
    for which, gr in enumerate(grads):
        for idx in np.ndindex(gr.shape):
            x = [q, k, v]
            plus = [a.copy() for a in x]
            minus = [a.copy() for a in x]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(fd - gr[idx]) < 1e-8
