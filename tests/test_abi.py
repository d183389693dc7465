"""The C-ABI library builds for sm_103a, loads, exports every entry point the
headers declare, and rejects bad arguments on the host before touching the GPU.
No compute call is made here."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_61_gb300 import attn, build
    build.build()
    return attn.load()


def _declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_the_forward():
    names = _declared_symbols()
    for n in ("attn_fwd", "attn_fwd_checked", "attn_strerror", "attn_last_cuda_error",
              "attn_device_error_info", "attn_probe_tile"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_library_targets_sm103a():
    from exact_attention_61_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in " ".join(build.ARCH)


def test_strerror(lib):
    from exact_attention_61_gb300 import attn
    for st in range(6):
        assert attn.strerror(st)
    assert attn.strerror(99) == "unknown status"


A = 1 << 20  # fake, 16-byte-aligned addresses: validation must reject before any CUDA call


def _call(lib_mod, **kw):
    args = dict(q=A, k=2 * A * 64, v=3 * A * 64, o=4 * A * 64, lse=5 * A * 64, B=1, H=2, N=128,
                d=64, causal=0, scale=0.125, dtype=1, stream=None)
    args.update(kw)
    return lib_mod.attn_fwd(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1), (dict(lse=0), 1),
    (dict(B=0), 1), (dict(H=0), 1), (dict(N=0), 1), (dict(N=-5), 1), (dict(d=0), 1),
    (dict(dtype=2), 1), (dict(dtype=-1), 1),
    (dict(scale=0.0), 1), (dict(scale=-0.5), 1), (dict(scale=float("inf")), 1),
    (dict(scale=float("nan")), 1),
    (dict(d=96), 2), (dict(d=32), 2), (dict(d=256), 2),
    (dict(q=A + 8), 3), (dict(o=4 * A * 64 + 2), 3), (dict(lse=5 * A * 64 + 4), 3),
    (dict(B=1 << 31), 2), (dict(B=1 << 16, H=1 << 16), 2),
    (dict(o=A), 1),                     # o aliases q
    (dict(lse=A + 4096), 1),            # lse overlaps q
    (dict(o=4 * A * 64, lse=4 * A * 64 + 16), 1),  # lse inside o
])
def test_host_validation(lib, kw, status):
    from exact_attention_61_gb300 import attn
    assert _call(attn, **kw) == status
    assert attn.attn_fwd_checked(**{**dict(q=A, k=2 * A * 64, v=3 * A * 64, o=4 * A * 64,
                                           lse=5 * A * 64, B=1, H=2, N=128, d=64, causal=0,
                                           scale=0.125, dtype=1, stream=None), **kw}) == status


def test_probe_validation(lib):
    f = lib.attn_probe_tile
    assert f(None, A, A, A, A, A, 64, 1, None) == 1
    assert f(A, A, A, A, A, A, 96, 1, None) == 2
    assert f(A, A, A, A + 4, A, A, 64, 1, None) == 3
    assert f(A, A, A, A, A, A, 64, 7, None) == 1
