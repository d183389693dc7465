"""Host-side arithmetic about the attention forward: FLOP convention, the causal
tile-skipping schedule, and memory-traffic models. Used by the benchmark to
report algorithmic and executed work, and pinned by tests against the numbers
the profile-driven FlashAttention-2 page prints.

All formulas restate "如何用 profiler 逐步优化 Triton FlashAttention-2 kernel"
(the profile-driven FlashAttention-2 page):
 * Round 0 / Step 5 ("The operations"): the algorithm needs 4*(B*H)*N^2*D
   FLOPs; Round 2 / Step 6: causal attention needs half of that.
 * Round 4 / Causal tile-skipping: per query tile starting at q_start, key
   tiles [0, unmasked_stop) need no mask and [unmasked_stop, masked_stop)
   straddle the diagonal (or a ragged end) and are masked; nothing past
   masked_stop is visited.
 * Round 0 / Step 5 ("The bytes"): L2 -> SM traffic = programs x (K and V of
   the head) plus each program's own Q tile.
"""
from __future__ import annotations

import math
from typing import Dict, Tuple


def attn_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Algorithmic FLOPs of the forward: 4*B*H*N^2*d, halved under the causal mask."""
    f = 4.0 * B * H * N * N * d
    return f / 2.0 if causal else f


def attn_exps(B: int, H: int, N: int, causal: bool) -> float:
    """Exponentials the softmax needs: one per visible score (B*H*N^2, halved if causal)."""
    e = float(B) * H * N * N
    return e / 2.0 if causal else e


def key_ranges(q_start: int, q_tile: int, k_tile: int, n_keys: int, causal: bool) -> Tuple[int, int]:
    """(unmasked_stop, masked_stop) in keys for the query tile starting at q_start."""
    full_stop = (n_keys // k_tile) * k_tile
    if causal:
        unmasked_stop = min((q_start // k_tile) * k_tile, full_stop)
        masked_stop = min(q_start + q_tile, n_keys)
    else:
        unmasked_stop = full_stop
        masked_stop = n_keys
    return unmasked_stop, masked_stop


def tile_pairs(N: int, q_tile: int, k_tile: int, causal: bool) -> Dict[str, int]:
    """Per head: how many (query tile, key tile) pairs the split loops visit."""
    total = math.ceil(N / q_tile) * math.ceil(N / k_tile)
    unmasked = masked = 0
    for q_start in range(0, N, q_tile):
        u, m = key_ranges(q_start, q_tile, k_tile, N, causal)
        unmasked += u // k_tile
        masked += math.ceil((m - u) / k_tile) if m > u else 0
    return {"total": total, "visited": unmasked + masked, "unmasked": unmasked, "masked": masked}


def executed_flops(B: int, H: int, N: int, d: int, q_tile: int, k_tile: int, causal: bool) -> float:
    """Tensor-core FLOPs actually issued when every visited tile pair is computed whole."""
    pairs = tile_pairs(N, q_tile, k_tile, causal)["visited"]
    return 4.0 * B * H * pairs * q_tile * k_tile * d


def l2_read_bytes(B: int, H: int, N: int, d: int, rows_per_program: int, elt_bytes: int = 2) -> float:
    """L2 -> SM bytes when every program reads all of K and V of its head once
    (non-causal) plus its own query rows."""
    programs = math.ceil(N / rows_per_program) * B * H
    kv = 2.0 * N * d * elt_bytes
    q = float(B) * H * N * d * elt_bytes
    return programs * kv + q


def min_hbm_bytes(B: int, H: int, N: int, d: int, elt_bytes: int = 2) -> float:
    """Compulsory DRAM traffic: read Q, K, V once, write O and the fp32 LSE once."""
    return 4.0 * B * H * N * d * elt_bytes + 4.0 * B * H * N


# ---- this library's kernel -----------------------------------------------------------------

KERNEL_Q_TILE = 128       # query rows per TMEM tile (one softmax warpgroup)
KERNEL_K_TILE = 128       # keys per K/V tile
KERNEL_ROWS_PER_CTA = 256  # two Q tiles share every K/V tile a CTA loads


def kernel_tile_pairs(N: int, causal: bool) -> int:
    """(128-row Q tile, 128-key tile) pairs the forward kernel computes per head."""
    return tile_pairs(N, KERNEL_Q_TILE, KERNEL_K_TILE, causal)["visited"]


def kernel_executed_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    return executed_flops(B, H, N, d, KERNEL_Q_TILE, KERNEL_K_TILE, causal)


def kernel_ctas(B: int, H: int, N: int) -> int:
    return math.ceil(N / KERNEL_ROWS_PER_CTA) * B * H
