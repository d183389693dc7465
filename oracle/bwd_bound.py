"""Per-element error bound of the 16-bit backward pass against the fp64 oracle.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: used by ``tests/`` and
``__graft_entry__.smoke()`` to judge a backward computed elsewhere.

The pages state no backward tolerance ("如何用 profiler 逐步优化 Triton
FlashAttention-2 kernel", "Future articles", only names the FA2 backward that
consumes L), so the bound follows the arithmetic of a 16-bit path with fp32
accumulation. With u the unit roundoff of the dtype (2^-11 fp16, 2^-8 bf16) and
g = n 2^-24 for fp32 sums over n terms:

- P is rounded to the dtype before dV += P^T dO, and dS before dK and dQ;
- D = dO . O is formed from the 16-bit O, so it is off by at most
  dD_i = sum_t |dO_it| (|O_used_it - O_it| + u |O_it|), and dS_ij by P_ij dD_i;
- each output is rounded once to the dtype.

  bound(dV) = (u + g) |P|^T |dO| + u |dV|
  bound(dK) = scale ((u + g) |dS| + P dD)^T |Q| + u |dK|
  bound(dQ) = scale ((u + g) |dS| + P dD) |K| + u |dQ|

An element passes within twice its bound plus 1e-6 absolute (for exact zeros).
"""
from __future__ import annotations

import numpy as np

U = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


def d_error(do64, o_used, o_exact, u):
    """Bound on |D_used - D| when D = dO . O is formed from o_used instead of the exact O."""
    return (np.abs(do64) * (np.abs(o_used - o_exact) + u * np.abs(o_exact))).sum(-1)


def bounds(ref, m, q64, k64, do64, dD, scale, dtype, n_keys):
    """Per-element bounds of dq, dk, dv. ref: oracle gradients {dq, dk, dv}; m: the
    materialised backward (its P and dS); dD: d_error(...) per query row."""
    u = U[dtype]
    g = n_keys * 2.0 ** -24
    p, ds = m["p"], m["ds"]
    eds = (u + g) * np.abs(ds) + p * dD[..., None]
    return {
        "dv": (u + g) * np.einsum("bhij,bhid->bhjd", p, np.abs(do64)) + u * np.abs(ref["dv"]),
        "dk": scale * np.einsum("bhij,bhid->bhjd", eds, np.abs(q64)) + u * np.abs(ref["dk"]),
        "dq": scale * np.einsum("bhij,bhjd->bhid", eds, np.abs(k64)) + u * np.abs(ref["dq"]),
    }


def check(got, ref, bnd):
    """(ok, message): every element of got[key] (fp64 arrays) within 2 * bound + 1e-6
    of ref[key], for key in dq, dk, dv."""
    for key in ("dq", "dk", "dv"):
        x = np.asarray(got[key], dtype=np.float64)
        if not np.isfinite(x).all():
            return False, f"non-finite {key}"
        err = np.abs(x - ref[key])
        lim = 2.0 * bnd[key] + 1e-6
        bad = err > lim
        if bad.any():
            return False, (f"{key}: {int(bad.sum())} elements over the bound; worst err {err.max():.3e}, "
                           f"at the worst element err/bound = {(err / lim).max():.2f}")
    return True, "ok"
