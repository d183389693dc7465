"""Seeded synthetic attention inputs.

This module is the only code that both the fp64 oracle tests and the CUDA-path
tests import. It draws numbers and rounds them to the storage dtype; it holds
none of the attention arithmetic.

Recipe (the pages only ever feed random normal tensors to their kernels:
"How I profile" and "The sweep" on the profile-driven FlashAttention-2 page,
and the correctness grid on the gpu-attention-phase1-phase2 page):

* one CPU ``torch.Generator`` seeded per workload, drawing Q, then K, then V,
  each ``randn`` in fp32 with shape ``[B, H, N, d]``;
* an optional exact multiply by a power of two (the wide-head long-sequence
  workload uses 2, to push the running row maximum around);
* one round-to-nearest-even cast to fp16 or bf16.

The rounded 16-bit tensors are what both sides consume.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import torch

_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


def to_dtype(name: str) -> torch.dtype:
    try:
        return _DTYPES[name]
    except KeyError:
        raise ValueError(f"unknown dtype {name!r}; expected one of {sorted(_DTYPES)}")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named problem: shapes, dtypes, masks, input scale and seed."""
    name: str
    B: int
    H: int
    N: int
    d: int
    dtypes: Tuple[str, ...]
    causal: Tuple[bool, ...]
    input_scale: float
    seed: int


# The fixed problems this library is measured and checked on. Seeds are fixed
# per problem so that every run draws the same tensors.
WORKLOADS: List[Workload] = [
    Workload("b1h1n128d64", 1, 1, 128, 64, ("fp16",), (False,), 1.0, 61000),
    Workload("b2h4n1000d64", 2, 4, 1000, 64, ("fp16", "bf16"), (False, True), 1.0, 61001),
    Workload("b4h16n4096d64", 4, 16, 4096, 64, ("bf16",), (False, True), 1.0, 61002),
    Workload("b1h16n8192d128x2", 1, 16, 8192, 128, ("bf16",), (True,), 2.0, 61003),
]


def workload(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


SWEEP_N = (512, 1024, 2048, 4096, 8192, 16384)
SWEEP_D = (64, 128)


def sweep_seed(N: int, d: int, dtype: str, causal: bool) -> int:
    """Seed of one sequence-sweep point, derived from its parameters."""
    return 61004 + 1000 * SWEEP_N.index(N) + 100 * SWEEP_D.index(d) + \
        10 * ("fp16", "bf16").index(dtype) + int(causal)


def sweep_points():
    """Every point of the sequence sweep: B = 16384/N, H = 16."""
    for N in SWEEP_N:
        for d in SWEEP_D:
            for dtype in ("fp16", "bf16"):
                for causal in (False, True):
                    yield dict(B=16384 // N, H=16, N=N, d=d, dtype=dtype, causal=causal,
                               seed=sweep_seed(N, d, dtype, causal))


def make_qkv(B: int, H: int, N: int, d: int, dtype: str, seed: int,
             input_scale: float = 1.0, generator: Optional[torch.Generator] = None):
    """Draw Q, K, V ~ N(0,1) (times ``input_scale``) in fp32 and round to ``dtype``.

    Returns three contiguous CPU tensors of shape [B, H, N, d].
    """
    g = generator if generator is not None else torch.Generator().manual_seed(int(seed))
    out = []
    for _ in range(3):
        x = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
        if input_scale != 1.0:
            x.mul_(input_scale)
        out.append(x.to(to_dtype(dtype)).contiguous())
    return tuple(out)


def make_qkv_rising(B: int, H: int, N: int, d: int, dtype: str, seed: int, step: float = 1.0):
    """Q, K, V whose scores rise along the keys, so that every 128-key tile raises the
    running row maximum by more than the kernel's lazy-rescale threshold (exercises the
    online rescaling on every tile).

    Q ~ N(0,1) + 1 and K[j] ~ N(0,1) + step * (j / 128) * 8 / sqrt(d) on every
    component; V ~ N(0,1). Drawn in fp32 from one seeded generator (Q, K, V in that
    order), then rounded to dtype.
    """
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((B, H, N, d), generator=g, dtype=torch.float32) + 1.0
    k = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
    ramp = torch.arange(N, dtype=torch.float32).div_(128.0).mul_(step * 8.0 / d ** 0.5)
    k.add_(ramp.view(1, 1, N, 1))
    dt = to_dtype(dtype)
    return q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous()


def make_qkv_kv(B: int, H: int, Nq: int, Nk: int, d: int, dtype: str, seed: int,
                input_scale: float = 1.0):
    """Q [B, H, Nq, d] and K, V [B, H, Nk, d], i.i.d. N(0,1) (times ``input_scale``).

    Same recipe as :func:`make_qkv` (one seeded generator, Q then K then V, fp32,
    one round-to-nearest-even cast) with separate query and key lengths, as in a
    KV-cache decode step (a few query rows against a long cache).
    """
    g = torch.Generator().manual_seed(int(seed))
    out = []
    for n in (Nq, Nk, Nk):
        x = torch.randn((B, H, n, d), generator=g, dtype=torch.float32)
        if input_scale != 1.0:
            x.mul_(input_scale)
        out.append(x.to(to_dtype(dtype)).contiguous())
    return tuple(out)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One KV-cache decode problem: Nq new query rows against an Nk-long cache."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    dtype: str
    seed: int


# Decode problems (the pages print no decode shapes; these are chosen to span a batch
# of single-token steps, a long single-sequence cache and a few-token speculative step).
DECODE_WORKLOADS: List[DecodeWorkload] = [
    DecodeWorkload("b8h32q1k8192d128", 8, 32, 1, 8192, 128, "bf16", 61100),
    DecodeWorkload("b1h16q1k65536d128", 1, 16, 1, 65536, 128, "bf16", 61101),
    DecodeWorkload("b16h16q4k4096d64", 16, 16, 4, 4096, 64, "fp16", 61102),
]


def decode_workload(name: str) -> DecodeWorkload:
    for w in DECODE_WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)
