"""Host-side counting arithmetic pinned to numbers the profile-driven
FlashAttention-2 page prints (tests/golden/fa2_profile_counts.txt)."""
import os

import pytest

from exact_attention_61_gb300 import counts

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fa2_profile_counts.txt")


def _golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv, where, prec = (x.strip() for x in line.split("|"))
            key, val = (x.strip() for x in kv.split("="))
            out[key] = (float(val), float(prec), where)
    return out


G = _golden()
B, H, N, D = 4, 8, 4096, 64


def _printed(name, got):
    """Compare with a value the page prints: exact for counts, else within the
    relative precision the printed digits carry."""
    want, prec, where = G[name]
    if prec == 0:
        assert got == want, f"{name}: {got} != {want} ({where})"
    else:
        assert abs(got - want) <= prec * want, f"{name}: {got} vs printed {want} ({where})"


def test_flop_convention():
    _printed("flops_noncausal", counts.attn_flops(B, H, N, D, False))
    _printed("flops_causal", counts.attn_flops(B, H, N, D, True))
    _printed("flops_duplicated_8warps", 2 * counts.attn_flops(B, H, N, D, False))


def test_causal_tile_pairs_64x32():
    p = counts.tile_pairs(N, 64, 32, causal=True)
    _printed("pairs_total_q64_k32", p["total"])
    _printed("pairs_visited_q64_k32", p["visited"])
    _printed("pairs_masked_q64_k32", p["masked"])
    _printed("pairs_unmasked_q64_k32", p["unmasked"])
    assert p["total"] - p["visited"] == 4032  # the fully masked pairs are never visited


def test_executed_ops_with_tile_skipping():
    got = counts.executed_flops(B, H, N, D, 64, 32, causal=True)
    _printed("executed_causal_q64_k32", got)
    waste = got / counts.attn_flops(B, H, N, D, True) - 1.0
    assert abs(waste - 0.016) < 0.001  # "+1.6% for the diagonal tiles"


def test_l2_traffic_model():
    _printed("l2_bytes_q16", counts.l2_read_bytes(B, H, N, D, 16))
    _printed("l2_bytes_q64", counts.l2_read_bytes(B, H, N, D, 64))


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 1000, 4096])
@pytest.mark.parametrize("qt,kt", [(64, 32), (128, 128), (64, 128), (16, 16)])
def test_ranges_cover_exactly_the_visible_keys(N, qt, kt):
    """Visited key tiles cover every visible key of every row, and the unmasked
    range holds only keys visible to every row of the query tile."""
    for causal in (False, True):
        for q_start in range(0, N, qt):
            u, m = counts.key_ranges(q_start, qt, kt, N, causal)
            assert u % kt == 0 and 0 <= u <= m <= N
            last_row = min(q_start + qt, N) - 1
            need = last_row + 1 if causal else N
            assert m >= need  # every visible key is visited
            if causal:
                assert u <= q_start  # keys below the tile's first row are visible to all rows
            assert u <= (N // kt) * kt  # unmasked tiles are whole tiles inside the sequence


def test_non_causal_has_no_skipped_tiles():
    p = counts.tile_pairs(1000, 128, 128, causal=False)
    assert p["visited"] == p["total"] == 64 and p["masked"] == 8
