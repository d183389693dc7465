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
    for st in range(7):
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


def test_headers_declare_the_kv_forward():
    names = _declared_symbols()
    for n in ("attn_fwd_kv", "attn_fwd_kv_checked", "attn_fwd_kv_workspace_bytes", "attn_bwd",
              "attn_bwd_checked", "attn_bwd_workspace_bytes", "attn_fwd_window",
              "attn_fwd_window_checked", "attn_bwd_window", "attn_bwd_window_checked"):
        assert n in names


def _call_kv(lib_mod, checked=False, **kw):
    args = dict(q=A, k=2 * A * 64, v=3 * A * 64, o=4 * A * 64, lse=5 * A * 64, B=1, H=2, Nq=4,
                Nk=1000, d=64, mask=2, scale=0.125, dtype=1, workspace=None, workspace_bytes=0,
                stream=None)
    args.update(kw)
    return lib_mod.attn_fwd_kv(**args, checked=checked)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), 1), (dict(Nq=0), 1), (dict(Nk=0), 1), (dict(Nk=-1), 1),
    (dict(mask=3), 1), (dict(mask=-1), 1), (dict(dtype=5), 1), (dict(scale=0.0), 1),
    (dict(d=80), 2), (dict(Nk=1 << 31), 2),
    (dict(k=2 * A * 64 + 8), 3), (dict(workspace=6 * A * 64 + 4, workspace_bytes=4096), 3),
    (dict(workspace=A, workspace_bytes=4096), 1),               # workspace overlaps q
    (dict(workspace=3 * A * 64 + 256, workspace_bytes=64), 1),  # workspace inside v
    (dict(o=2 * A * 64), 1),                                     # o aliases k
])
def test_kv_host_validation(lib, kw, status):
    from exact_attention_61_gb300 import attn
    assert _call_kv(attn, **kw) == status
    assert _call_kv(attn, checked=True, **kw) == status


def _splits(attn, B, H, Nq, Nk, d):
    """Key ranges of the tensor-core split (0: none), from its workspace bytes."""
    n = attn.plan_split_for(B * H, Nq, Nk, d, 1 << 40, 152)[2]
    per = B * H * Nq * (d + 1) * 4
    assert n % per == 0
    assert n <= attn.workspace_bytes(B, H, Nq, Nk, d)
    return n // per


@pytest.mark.parametrize("B,H,Nq,Nk,d", [
    (1, 8, 1, 8192, 128), (8, 32, 1, 32768, 64), (1, 1, 1, 128, 64), (1, 1, 1, 129, 64),
    (2, 4, 16, 65536, 128), (1, 16, 300, 20000, 64), (4, 16, 4096, 4096, 64), (1, 1, 5, 100, 64),
    (8, 32, 1, 8192, 128), (16, 16, 4, 4096, 64), (1, 16, 1, 65536, 128),
])
def test_workspace_split_plan(lib, B, H, Nq, Nk, d):
    """The split of the keys: none when the query rows already give two CTAs per SM of a
    152-SM GPU; otherwise the range count minimises ceil(CTAs * S / 152) waves of
    (tiles per range + 2) tile times over every count up to eight waves of CTAs, with no
    empty range (brute force over all counts here)."""
    from exact_attention_61_gb300 import attn
    ctas = -(-Nq // 256) * B * H
    n_kv = -(-Nk // 128)
    S = _splits(attn, B, H, Nq, Nk, d)
    if ctas >= 304:
        assert S == 0
        return

    def cost(c):
        t = -(-n_kv // c)
        return -(-ctas * -(-n_kv // t) // 152) * (t + 2)

    best = min(cost(c) for c in range(1, min(n_kv, -(-8 * 152 // ctas)) + 1))
    if S == 0:  # no split
        assert cost(1) == best
        return
    assert 2 <= S <= n_kv
    tps = -(-n_kv // S)
    assert (S - 1) * tps < n_kv <= S * tps  # no empty range
    assert cost(S) == best


def test_workspace_bytes_rejects_bad_sizes(lib):
    from exact_attention_61_gb300 import attn
    assert attn.workspace_bytes(0, 1, 1, 100, 64) == 0
    assert attn.workspace_bytes(1, 1, 1, 100, 96) == 0
    assert attn.workspace_bytes(1, 1, 1, 0, 64) == 0


def test_static_scratch_entry_rejects_before_any_cuda_call(lib):
    """attn_fwd_kv_static validates like attn_fwd_kv and refuses sizes whose split needs
    more than its 16 MiB static scratch, all on the host (fake pointers here)."""
    from exact_attention_61_gb300 import attn
    args = dict(q=A, k=2 * A * 64, v=3 * A * 64, o=4 * A * 64, lse=5 * A * 64, B=1, H=2, Nq=4,
                Nk=1000, d=64, mask=2, scale=0.125, dtype=1, stream=None)
    assert attn.attn_fwd_kv_static(**{**args, "q": 0}) == 1
    assert attn.attn_fwd_kv_static(**{**args, "mask": 7}) == 1
    assert attn.attn_fwd_kv_static(**{**args, "d": 96}) == 2
    assert attn.attn_fwd_kv_static(**{**args, "lse": 5 * A * 64 + 4}) == 3
    big = dict(B=1, H=64, Nq=256, Nk=65536, d=128)
    assert attn.workspace_bytes(**big) > attn.STATIC_SCRATCH_BYTES
    G = 1 << 32  # fake addresses far enough apart for these sizes
    spaced = dict(q=G, k=2 * G, v=3 * G, o=4 * G, lse=5 * G)
    assert attn.attn_fwd_kv_static(**{**args, **big, **spaced}) == attn.ATTN_ERR_SCRATCH_TOO_SMALL
    assert "static scratch" in attn.strerror(attn.ATTN_ERR_SCRATCH_TOO_SMALL)
    # every size with at most 16 query rows fits
    for BH in (1, 7, 100, 151, 152, 303):
        for d in (64, 128):
            assert attn.workspace_bytes(1, BH, 16, 1 << 20, d) <= attn.STATIC_SCRATCH_BYTES


def _call_bwd(attn, checked=False, **kw):
    M = 64 * A  # 64 MiB apart: room for every tensor of the default sizes
    args = dict(q=1 * M, k=2 * M, v=3 * M, o=4 * M, lse=5 * M, dout=6 * M, dq=7 * M, dk=8 * M,
                dv=9 * M, B=1, H=2, N=300, d=64, causal=1, scale=0.125, dtype=1, workspace=10 * M,
                workspace_bytes=1 << 20, stream=None)
    args.update(kw)
    return attn.attn_bwd(**args, checked=checked)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), 1), (dict(dout=0), 1), (dict(dq=0), 1), (dict(workspace=0), 1),
    (dict(N=0), 1), (dict(dtype=3), 1), (dict(scale=-1.0), 1),
    (dict(d=32), 2), (dict(B=1 << 31), 2),
    (dict(dk=8 * 64 * A + 8), 3), (dict(lse=5 * 64 * A + 4), 3), (dict(workspace=10 * 64 * A + 2), 3),
    (dict(workspace_bytes=100), 1),          # short workspace
    (dict(dq=64 * A), 1),                    # dq aliases q
    (dict(dk=7 * 64 * A), 1),                # dk aliases dq
    (dict(dv=64 * A + 4096), 1),             # dv inside q
    (dict(workspace=9 * 64 * A + 1024), 1),  # workspace overlaps dv
])
def test_bwd_host_validation(lib, kw, status):
    from exact_attention_61_gb300 import attn
    assert _call_bwd(attn, **kw) == status
    assert _call_bwd(attn, checked=True, **kw) == status


def test_bwd_workspace_bytes(lib):
    from exact_attention_61_gb300 import attn
    # 8 bytes per row padded to 128 rows (LSE, D) + 4 d bytes per row (dQ accumulator)
    # D and LSE vectors (rows padded to 128), the fp32 dQ accumulator, a 16-byte work counter
    assert attn.bwd_workspace_bytes(1, 2, 300, 64) == 2 * 384 * 8 + 2 * 300 * 64 * 4 + 16
    assert attn.bwd_workspace_bytes(4, 16, 4096, 128) == 64 * 4096 * 8 + 64 * 4096 * 128 * 4 + 16
    assert attn.bwd_workspace_bytes(1, 1, 1, 96) == 0
    assert attn.bwd_workspace_bytes(0, 1, 128, 64) == 0


def test_window_host_validation(lib):
    from exact_attention_61_gb300 import attn
    args = dict(q=A, k=2 * A * 64, v=3 * A * 64, o=4 * A * 64, lse=5 * A * 64, B=1, H=2, Nq=128, Nk=500,
                d=64, window_left=64, window_right=0, kv_lens=None, align=1, scale=0.125, dtype=1,
                workspace=None, workspace_bytes=0, stream=None)
    for checked in (False, True):
        f = lambda **kw: attn.attn_fwd_window(**{**args, **kw}, checked=checked)
        assert f(align=2) == 1
        assert f(align=-1) == 1
        assert f(kv_lens=6 * A * 64 + 2) == 3
        assert f(q=0) == 1
        assert f(d=80) == 2
        G = 1 << 40  # fake addresses far enough apart for 2^30 keys
        assert f(Nk=1 << 30, q=G, k=2 * G, v=3 * G, o=4 * G, lse=5 * G) == 2  # Nq + Nk beyond 2^30
        assert f(dtype=9) == 1


# ---- attn_fwd_host: host-side planning and validation (no CUDA call) ------------------------

def test_headers_declare_the_host_forward():
    names = _declared_symbols()
    for n in ("attn_fwd_host", "attn_fwd_host_checked", "attn_fwd_host_workspace_bytes", "attn_fwd_host_plan"):
        assert n in names


@pytest.mark.parametrize("B,H,N,d", [
    (4, 16, 4096, 64), (1, 1, 1, 64), (1, 1, 100, 128), (32, 16, 512, 64), (1, 16, 8192, 128),
    (2, 2, 777, 64), (64, 64, 128, 64), (1, 200, 65536, 128), (3, 5, 300, 128), (1024, 1, 256, 64),
])
def test_host_plan_covers_every_head(lib, B, H, N, d):
    from exact_attention_61_gb300 import attn
    n, h = attn.host_plan(B, H, N, d)
    BH = B * H
    ctiles = -(-N // 256)
    assert 1 <= n <= 16 and 1 <= h <= BH
    assert (n - 1) * h < BH <= n * h          # the chunks cover [0, BH) once; the last holds the rest
    if n > 1:
        # every chunk but the last fills two waves of one CTA per SM of a 152-SM GPU
        assert h * ctiles >= 2 * 152
    else:
        assert h == BH
    if h * ctiles > 2 * 152 + ctiles:
        assert n == 16 or h == BH                 # chunks grow past two waves only to stay <= 16


def test_host_workspace_layout(lib):
    from exact_attention_61_gb300 import attn
    up = lambda x: (x + 255) // 256 * 256
    for B, H, N, d in ((4, 16, 4096, 64), (1, 1, 1, 64), (2, 3, 77, 128)):
        X = up(B * H * N * d * 2)
        assert attn.host_workspace_bytes(B, H, N, d) == 4 * X + up(B * H * N * 4)
    for bad in ((0, 1, 1, 64), (1, 0, 1, 64), (1, 1, 0, 64), (1, 1, 1, 96), (1 << 31, 1, 1, 64)):
        assert attn.host_workspace_bytes(*bad) == 0
        assert attn.host_plan(*bad) == (0, 0)


W = 1 << 40  # fake device workspace address (256-byte aligned)


def _call_host(lib_mod, checked=False, **kw):
    B, H, N, d = kw.get("B", 1), kw.get("H", 2), kw.get("N", 128), kw.get("d", 64)
    ws_n = lib_mod.host_workspace_bytes(B, H, N, d) if d in (64, 128) and min(B, H, N) > 0 else 1 << 20
    args = dict(q=A, k=2 * A * 64, v=3 * A * 64, o=4 * A * 64, lse=5 * A * 64, B=B, H=H, N=N, d=d, causal=0,
                scale=0.125, dtype=1, workspace=W, workspace_bytes=ws_n, stream=None)
    args.update(kw)
    return lib_mod.attn_fwd_host(**args, checked=checked)


@pytest.mark.parametrize("kw,status", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(q=0, k=0), 1), (dict(k=0, v=0), 1),
    (dict(q=0, k=0, v=0, o=0), 1), (dict(q=0, k=0, v=0, lse=0), 1),
    (dict(o=0), 1), (dict(lse=0), 1), (dict(workspace=0), 1),
    (dict(B=0), 1), (dict(N=-1), 1), (dict(dtype=2), 1), (dict(scale=0.0), 1), (dict(scale=float("nan")), 1),
    (dict(d=96), 2), (dict(B=1 << 31), 2),
    (dict(workspace=W + 16), 3),                 # the workspace must be 256-byte aligned
    (dict(workspace_bytes=1000), 1),             # too small
    (dict(o=A), 1),                              # o aliases q
    (dict(lse=2 * A * 64 + 64), 1),              # lse inside k
    (dict(o=4 * A * 64, lse=4 * A * 64 + 512), 1),   # lse inside o
    (dict(q=W + 4096), 1),                       # an input inside the workspace
])
def test_host_entry_validation(lib, kw, status):
    from exact_attention_61_gb300 import attn
    assert _call_host(attn, **kw) == status
    assert _call_host(attn, checked=True, **kw) == status


def test_host_entry_accepts_unaligned_host_buffers(lib):
    """Host buffers need no alignment: an odd address passes validation and the call only
    fails later, at the CUDA query of the (fake) workspace, with ATTN_ERR_CUDA."""
    from exact_attention_61_gb300 import attn
    assert _call_host(attn, q=A + 3, o=4 * A * 64 + 1) == attn.ATTN_ERR_CUDA


def test_host_entry_staged_inputs_pass_validation(lib):
    """q = k = v = NULL (inputs already staged in the workspace) is valid: the call gets as far
    as the CUDA query of the (fake) workspace and fails there with ATTN_ERR_CUDA."""
    from exact_attention_61_gb300 import attn
    assert _call_host(attn, q=0, k=0, v=0) == attn.ATTN_ERR_CUDA
    assert _call_host(attn, q=0, k=0, v=0, workspace=W + 16) == attn.ATTN_ERR_MISALIGNED
    assert _call_host(attn, q=0, k=0, v=0, o=W + 256) == attn.ATTN_ERR_INVALID_ARG   # o inside the workspace


def test_planners_follow_the_sm_count(lib):
    """The split of the keys (attn_fwd_kv) and the chunks of heads (attn_fwd_host) are
    planned for the SM count of the GPU they run on: the test hooks take it as an argument.
    Without a device the public queries plan for a GB300's 152 SMs."""
    from exact_attention_61_gb300 import attn
    # chunks of about two waves of 256-row items: ceil(2 * SMs / ceil(N / 256)) heads
    assert attn.plan_host_for(64, 4096, 152) == (4, 19)
    assert attn.plan_host_for(64, 4096, 76) == (7, 10)
    assert attn.plan_host_for(64, 4096, 304) == (2, 38)
    assert attn.plan_host_for(64, 4096, 152) == attn.host_plan(4, 16, 4096, 64)
    # decode: 8 x 32 single-row heads against 8192 keys are 256 CTAs
    full = 1 << 40
    n152, tps152, b152 = attn.plan_split_for(256, 1, 8192, 128, full, 152)
    assert n152 == 4 and tps152 == 16 and b152 == 256 * 4 * 1 * 129 * 4
    # (one query row: the streaming decode kernel runs; the query leaves room for both plans)
    assert b152 <= attn.workspace_bytes(8, 32, 1, 8192, 128)
    assert attn.plan_split_for(256, 1, 8192, 128, full, 76)[0] == 1   # 256 CTAs already fill 76 SMs twice
    # 304 SMs hold the 256 CTAs in one wave (no split); 2048 SMs make room for more ranges
    assert attn.plan_split_for(256, 1, 8192, 128, full, 304)[0] == 1
    assert attn.plan_split_for(256, 1, 8192, 128, full, 2048)[0] > n152
    # a workspace that holds three ranges caps the split below the full plan's four
    assert attn.plan_split_for(256, 1, 8192, 128, 3 * 256 * 129 * 4, 152)[0] <= 3
    for sms in (1, 16, 132, 148, 152, 160, 200):
        for BH, Nq, Nk in ((1, 1, 65536), (16, 4, 4096), (300, 16, 1 << 20), (5, 300, 777)):
            n, tps, nbytes = attn.plan_split_for(BH, Nq, Nk, 64, full, sms)
            n_kv = (Nk + 127) // 128
            assert 1 <= n <= n_kv and tps * n >= n_kv and tps * (n - 1) < n_kv
            assert nbytes == (0 if n == 1 else BH * n * Nq * 65 * 4)
            if Nq <= 16:
                assert nbytes <= attn.STATIC_SCRATCH_BYTES


def test_decode_planner(lib):
    """The streaming decode kernel's plan: key ranges of whole 32-key tiles covering every
    key, the workspace the partials need (none for one range), at most one CTA per SM,
    capped by the workspace, and the plans of the three decode workloads on 152 SMs."""
    from exact_attention_61_gb300 import attn
    full = 1 << 40
    # (BH, Nq, Nk, d) -> (ranges, keys per range)
    assert attn.plan_decode_for(256, 1, 8192, 128, full, 152)[:2] == (7, 1184)
    assert attn.plan_decode_for(16, 1, 65536, 128, full, 152)[:2] == (38, 1728)
    assert attn.plan_decode_for(256, 4, 4096, 64, full, 152)[:2] == (7, 608)
    for sms in (1, 16, 132, 148, 152, 200):
        for BH, Nq, Nk, d in ((1, 1, 1, 64), (1, 1, 65536, 128), (256, 4, 4096, 64), (300, 3, 1 << 20, 64),
                              (5, 2, 777, 128), (4096, 1, 100, 128)):
            n, rk, grid, nbytes = attn.plan_decode_for(BH, Nq, Nk, d, full, sms)
            assert rk % 32 == 0 and rk * (n - 1) < Nk <= rk * n
            assert nbytes == (0 if n == 1 else BH * n * Nq * (d + 1) * 4)
            warps = 4 if d == 128 else (8 if Nq == 1 else 12)
            assert 1 <= grid <= sms and grid == min(sms, -(-BH * n // warps))
            assert nbytes <= attn.workspace_bytes(1, BH, Nq, Nk, d) or sms != 152
    # the workspace caps the ranges; no workspace: one range, O written directly
    cap = 3 * 256 * 129 * 4
    assert attn.plan_decode_for(256, 1, 8192, 128, cap, 152)[0] <= 3
    assert attn.plan_decode_for(256, 1, 8192, 128, 0, 152)[0::3] == (1, 0)
    with pytest.raises(attn.AttnError):
        attn.plan_decode_for(2, 5, 100, 64, full, 152)  # more rows than the decode kernel takes
