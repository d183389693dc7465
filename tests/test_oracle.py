"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these calls the CUDA path. Each pin is chosen so that a plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand, the wrong mask direction, the wrong log base, a missing scale) fails
at least one of them; ``test_pins_catch_planted_mistakes`` plants such mistakes
in copies of the oracle and checks exactly that.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gen import make_qkv

TIGHT = 1e-12


def _rand64(B, H, N, d, seed):
    g = np.random.default_rng(seed)
    return tuple(g.standard_normal((B, H, N, d)) for _ in range(3))


# --- brute force: the whole score matrix ---------------------------------------------------

@pytest.mark.parametrize("N", [1, 2, 7, 64, 129, 256])
@pytest.mark.parametrize("d", [1, 3, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_definition_matches_materialised(N, d, causal):
    q, k, v = _rand64(2, 2, N, d, seed=N * 31 + d)
    o, lse = oracle.attn_fwd(q, k, v, causal)
    o2, lse2 = oracle.attn_fwd_materialised(q, k, v, causal)
    np.testing.assert_allclose(o, o2, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=TIGHT)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_definition_matches_torch_sdpa_fp64(dtype, causal):
    """Independent library cross-check: torch CPU float64 SDPA and logsumexp."""
    q, k, v = make_qkv(2, 3, 200, 64, dtype, seed=7)
    scale = 0.125
    o, lse = oracle.attn_fwd(q, k, v, causal, scale)
    q64, k64, v64 = (t.to(torch.float64) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(q64, k64, v64, is_causal=causal,
                                                           scale=scale)
    s = scale * (q64 @ k64.transpose(-1, -2))
    if causal:
        s = s.masked_fill(~torch.ones(200, 200, dtype=torch.bool).tril(), float("-inf"))
    ref_lse = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-12)


# --- algebraic identity: the tiled online softmax equals the definition --------------------

@pytest.mark.parametrize("block", [1, 37, 128, 300])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tau", [0.0, 8.0])
def test_online_softmax_equals_definition(block, causal, tau):
    q, k, v = _rand64(1, 2, 300, 16, seed=block)
    q *= 3.0  # a wide spread of scores so the running maximum moves
    o, lse = oracle.attn_fwd(q, k, v, causal)
    o2, lse2 = oracle.attn_fwd_online(q, k, v, causal, block=block, tau=tau)
    np.testing.assert_allclose(o2, o, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=TIGHT)


# --- closed forms and invariants -----------------------------------------------------------

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_causal_row0_is_v0(dtype):
    """Under the causal mask row 0 sees only key 0: softmax of one value is 1,
    so O[0] = V[0] and LSE[0] = scale*q0.k0 (phase-1/2 page, Phase 1)."""
    q, k, v = make_qkv(2, 2, 50, 64, dtype, seed=3)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.125)
    v64, q64, k64 = (oracle.to_f64(t) for t in (v, q, k))
    np.testing.assert_array_equal(o[:, :, 0], v64[:, :, 0])
    expect = 0.125 * np.einsum("bhd,bhd->bh", q64[:, :, 0], k64[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], expect, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_scores_give_mean_of_v(causal):
    """Q = 0 makes every visible score 0: O[i] is the mean of the visible V rows
    and LSE[i] = ln |V_i| (natural log)."""
    N, d = 40, 8
    _, k, v = _rand64(1, 1, N, d, seed=11)
    q = np.zeros_like(k)
    o, lse = oracle.attn_fwd(q, k, v, causal, 0.3)
    for i in range(N):
        n_vis = i + 1 if causal else N
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n_vis].mean(axis=0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(n_vis)) < 1e-14


def test_single_key_gives_v():
    q, k, v = _rand64(3, 2, 1, 64, seed=5)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.2)
        np.testing.assert_array_equal(o, v)
        np.testing.assert_allclose(lse, 0.2 * np.einsum("bhnd,bhnd->bhn", q, k), atol=1e-13)


def test_two_keys_logistic_form():
    """Two keys with scaled scores a and b: the weight of key 0 is the logistic
    function of a - b, and LSE = max(a,b) + log1p(exp(-|a-b|))."""
    g = np.random.default_rng(2)
    for _ in range(20):
        d = 4
        q = g.standard_normal((1, 1, 1, d))
        k = g.standard_normal((1, 1, 2, d))
        v = g.standard_normal((1, 1, 2, d))
        q_rep = np.repeat(q, 2, axis=2)  # same query in both rows, non-causal
        o, lse = oracle.attn_fwd(q_rep, k, v, False, 0.7)
        a = 0.7 * float(q[0, 0, 0] @ k[0, 0, 0])
        b = 0.7 * float(q[0, 0, 0] @ k[0, 0, 1])
        w0 = 1.0 / (1.0 + math.exp(b - a))
        np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 1] + w0 * (v[0, 0, 0] - v[0, 0, 1]),
                                   atol=1e-14)
        assert abs(lse[0, 0, 0] - (max(a, b) + math.log1p(math.exp(-abs(a - b))))) < 1e-13


def test_key_permutation_invariance():
    """Without a mask, reordering keys together with their values changes nothing."""
    q, k, v = _rand64(1, 2, 77, 16, seed=9)
    perm = np.random.default_rng(1).permutation(77)
    o, lse = oracle.attn_fwd(q, k, v, False)
    o2, lse2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], False)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)


def test_constant_key_shift():
    """Adding one vector u to every key adds scale*q_i.u to every score of row i:
    O is unchanged and LSE shifts by scale*q_i.u."""
    q, k, v = _rand64(1, 1, 60, 8, seed=21)
    u = np.random.default_rng(4).standard_normal(8)
    o, lse = oracle.attn_fwd(q, k, v, False, 0.5)
    o2, lse2 = oracle.attn_fwd(q, k + u, v, False, 0.5)
    np.testing.assert_allclose(o2, o, atol=1e-12)
    np.testing.assert_allclose(lse2, lse + 0.5 * (q[0, 0] @ u), atol=1e-12)


def test_causal_row_ignores_future_keys():
    """Under the causal mask, changing key/value j > i leaves row i unchanged, and
    changing key/value j <= i changes it."""
    q, k, v = _rand64(1, 1, 30, 8, seed=13)
    o, _ = oracle.attn_fwd(q, k, v, True)
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, 20] += 5.0
    v2[0, 0, 20] += 5.0
    o2, _ = oracle.attn_fwd(q, k2, v2, True)
    np.testing.assert_array_equal(o2[0, 0, :20], o[0, 0, :20])
    assert np.abs(o2[0, 0, 20:] - o[0, 0, 20:]).max() > 1e-3


def test_rows_match_full():
    q, k, v = _rand64(2, 3, 90, 16, seed=17)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal)
        rows = np.array([0, 1, 89, 90, 179, 200, 539])
        o2, lse2 = oracle.attn_fwd_rows(q, k, v, causal, rows)
        np.testing.assert_array_equal(o2, o.reshape(-1, 16)[rows])
        np.testing.assert_array_equal(lse2, lse.reshape(-1)[rows])


def test_convex_combination_bounds():
    """Every output is a convex combination of visible V rows: all-ones V gives
    all-ones O, and each O[i,t] lies within the range of V[:, t] over V_i."""
    q, k, v = _rand64(1, 2, 50, 4, seed=23)
    o, _ = oracle.attn_fwd(q, k, np.ones_like(v), True)
    np.testing.assert_allclose(o, 1.0, atol=1e-14)
    o, _ = oracle.attn_fwd(q, k, v, True)
    for i in range(50):
        lo = v[:, :, :i + 1].min(axis=2)
        hi = v[:, :, :i + 1].max(axis=2)
        assert np.all(o[:, :, i] >= lo - 1e-12) and np.all(o[:, :, i] <= hi + 1e-12)


def test_bad_arguments_rejected():
    q, k, v = _rand64(1, 1, 4, 4, seed=0)
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, v, False, scale=0.0)
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, v, False, scale=-1.0)
    with pytest.raises(ValueError):
        oracle.attn_fwd_rows(q, k, v, False, rows=[4])


# --- the pins above catch plausible mistakes ------------------------------------------------

def _mutant_forward(q, k, v, causal, scale, mistake):
    """A copy of the materialised oracle with one planted mistake."""
    q64, k64, v64 = oracle.to_f64(q), oracle.to_f64(k), oracle.to_f64(v)
    N = q64.shape[2]
    sc = 1.0 if mistake == "no_scale" else scale
    kk = k64
    s = sc * np.einsum("bhid,bhjd->bhij", q64, kk)
    if causal:
        keep = np.tril(np.ones((N, N), dtype=bool), k=-1 if mistake == "strict_mask" else 0)
        if mistake == "upper_mask":
            keep = np.triu(np.ones((N, N), dtype=bool))
        s = np.where(keep, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    if mistake == "v_transposed_index":
        o = np.einsum("bhij,bhjd->bhid", e, v64[:, :, ::-1]) / l
    else:
        o = np.einsum("bhij,bhjd->bhid", e, v64) / l
    if mistake == "drop_norm":
        o = o * l
    lse = (m + (np.log2(l) if mistake == "log2_lse" else np.log(l)))[..., 0]
    if mistake == "lse_without_max":
        lse = np.log(l)[..., 0]
    return o, lse


def _pins_pass(fwd):
    """The closed-form pins above, applied to an arbitrary forward function."""
    ok = True
    q, k, v = _rand64(1, 1, 12, 4, seed=31)
    o, lse = fwd(q, k, v, True, 0.5)
    ok &= bool(np.allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-12))
    ok &= bool(abs(lse[0, 0, 0] - 0.5 * q[0, 0, 0] @ k[0, 0, 0]) < 1e-12)
    z = np.zeros_like(q)
    o, lse = fwd(z, k, v, True, 0.5)
    for i in range(12):
        ok &= bool(np.allclose(o[0, 0, i], v[0, 0, :i + 1].mean(axis=0), atol=1e-12))
        ok &= bool(abs(lse[0, 0, i] - math.log(i + 1)) < 1e-12)
    o1, l1 = fwd(q[:, :, :1], k[:, :, :1], v[:, :, :1], False, 0.5)
    ok &= bool(np.allclose(o1, v[:, :, :1], atol=1e-12))
    ok &= bool(np.allclose(l1[0, 0, 0], 0.5 * q[0, 0, 0] @ k[0, 0, 0], atol=1e-12))
    ref_o, ref_l = oracle.attn_fwd_materialised(q, k, v, False, 0.5)
    o, lse = fwd(q, k, v, False, 0.5)
    ok &= bool(np.allclose(o, ref_o, atol=1e-12) and np.allclose(lse, ref_l, atol=1e-12))
    return ok


@pytest.mark.parametrize("mistake", ["no_scale", "strict_mask", "upper_mask",
                                     "v_transposed_index", "drop_norm", "log2_lse",
                                     "lse_without_max"])
def test_pins_catch_planted_mistakes(mistake):
    assert _pins_pass(lambda *a: oracle.attn_fwd_materialised(*a))
    assert _pins_pass(lambda *a: oracle.attn_fwd(*a))
    assert not _pins_pass(lambda q, k, v, c, s: _mutant_forward(q, k, v, c, s, mistake))


# --- Nq query rows against Nk keys (decode and cross lengths) -------------------------------

@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 10), (5, 15), (1, 64), (7, 300), (64, 64), (40, 25)])
@pytest.mark.parametrize("causal", [False, True])
def test_qk_matches_materialised(Nq, Nk, causal):
    """Includes the shapes of "Programming an attention kernel in Triton", Kernel 4:
    Q (5, 32) against K/V (15, 32), and a single query (1, 64) against (10, 64)."""
    g = np.random.default_rng(Nq * 1000 + Nk)
    d = 32
    q = g.standard_normal((2, 2, Nq, d))
    k = g.standard_normal((2, 2, Nk, d))
    v = g.standard_normal((2, 2, Nk, d))
    o, lse = oracle.attn_fwd_qk(q, k, v, causal, 0.3)
    o2, lse2 = oracle.attn_fwd_qk_materialised(q, k, v, causal, 0.3)
    np.testing.assert_allclose(o, o2, rtol=0, atol=TIGHT)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lse2))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse[fin], lse2[fin], rtol=0, atol=TIGHT)


@pytest.mark.parametrize("Nq,Nk", [(3, 50), (1, 128), (20, 20)])
@pytest.mark.parametrize("causal", [False, True])
def test_qk_matches_torch_sdpa_explicit_mask(Nq, Nk, causal):
    """Independent library check with an explicit boolean mask (torch's own is_causal
    aligns top-left for Nq != Nk, so the bottom-right mask is spelled out)."""
    q, _, _ = make_qkv(1, 2, Nq, 64, "bf16", seed=Nq)
    _, k, v = make_qkv(1, 2, Nk, 64, "bf16", seed=Nk + 1)
    o, lse = oracle.attn_fwd_qk(q, k, v, causal, 0.125)
    q64, k64, v64 = (t.to(torch.float64) for t in (q, k, v))
    mask = torch.ones(Nq, Nk, dtype=torch.bool)
    if causal:
        mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
    ref = torch.nn.functional.scaled_dot_product_attention(q64, k64, v64, attn_mask=mask, scale=0.125)
    s = (0.125 * (q64 @ k64.transpose(-1, -2))).masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def test_qk_reduces_to_square_and_last_row_sees_all():
    q, k, v = _rand64(1, 2, 33, 8, seed=41)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal)
        o2, lse2 = oracle.attn_fwd_qk(q, k, v, causal)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(lse, lse2)
    # decode: the last query row under the bottom-right causal mask sees every key
    g = np.random.default_rng(3)
    qd = g.standard_normal((1, 1, 4, 8))
    oc, lc = oracle.attn_fwd_qk(qd, k[:, :1], v[:, :1], True)
    on, ln = oracle.attn_fwd_qk(qd, k[:, :1], v[:, :1], False)
    np.testing.assert_array_equal(oc[:, :, -1], on[:, :, -1])
    np.testing.assert_array_equal(lc[:, :, -1], ln[:, :, -1])
    # and row i sees exactly i + Nk - Nq + 1 keys: zero queries give the mean of those
    z = np.zeros((1, 1, 4, 8))
    oz, lz = oracle.attn_fwd_qk(z, k[:, :1], v[:, :1], True)
    for i in range(4):
        n_vis = i + 33 - 4 + 1
        np.testing.assert_allclose(oz[0, 0, i], v[0, 0, :n_vis].mean(axis=0), atol=1e-14)
        assert abs(lz[0, 0, i] - math.log(n_vis)) < 1e-14


@pytest.mark.parametrize("Nq,Nk", [(1, 10), (5, 15), (40, 25), (300, 7), (64, 64)])
def test_qk_top_left_matches_materialised(Nq, Nk):
    g = np.random.default_rng(Nq * 7 + Nk)
    q = g.standard_normal((1, 3, Nq, 16))
    k = g.standard_normal((1, 3, Nk, 16))
    v = g.standard_normal((1, 3, Nk, 16))
    o, lse = oracle.attn_fwd_qk(q, k, v, True, 0.4, align="top_left")
    o2, lse2 = oracle.attn_fwd_qk_materialised(q, k, v, True, 0.4, align="top_left")
    np.testing.assert_allclose(o, o2, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=TIGHT)


@pytest.mark.parametrize("Nq,Nk", [(3, 50), (50, 3), (17, 130)])
def test_qk_top_left_matches_torch_is_causal(Nq, Nk):
    """torch's SDPA with is_causal=True keeps the top-left alignment for Nq != Nk, so
    it pins the top-left mode without spelling the mask out."""
    q, _, _ = make_qkv(1, 2, Nq, 64, "fp16", seed=Nq + 5)
    _, k, v = make_qkv(1, 2, Nk, 64, "fp16", seed=Nk + 6)
    o, _ = oracle.attn_fwd_qk(q, k, v, True, 0.125, align="top_left")
    q64, k64, v64 = (t.to(torch.float64) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(q64, k64, v64, is_causal=True, scale=0.125)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    # the two alignments differ whenever Nq != Nk
    ob, _ = oracle.attn_fwd_qk(q, k, v, True, 0.125, align="bottom_right")
    assert np.abs(ob - o).max() > 1e-3


def test_qk_rows_without_keys():
    """More query rows than keys under the causal mask: the first Nq - Nk rows see no
    key and get O = 0, LSE = -inf; the others see keys up to their diagonal."""
    q, _, _ = _rand64(1, 1, 6, 4, seed=8)
    _, k, v = _rand64(1, 1, 2, 4, seed=9)
    o, lse = oracle.attn_fwd_qk(q, k, v, True)
    assert np.all(o[0, 0, :4] == 0) and np.all(np.isneginf(lse[0, 0, :4]))
    np.testing.assert_allclose(o[0, 0, 4], v[0, 0, 0], atol=1e-15)
    assert np.isfinite(lse[0, 0, 5])
