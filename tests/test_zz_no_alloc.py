"""attn_fwd_kv_static, the entry point that allocates nothing (split partials in the
library's static device scratch), against attn_fwd_kv with a caller workspace.

Collected last on purpose: it must pass alone and after every other test, i.e. with
whatever the earlier calls left in the static scratch. Two calls in a row on
different inputs each match attn_fwd_kv within the parity tolerances (O max-abs 4e-3
fp16 / 3.2e-2 bf16, LSE 1e-3).
"""
import pytest
import torch

from gen import DECODE_WORKLOADS, make_qkv_kv

TOL_O = {"fp16": 4e-3, "bf16": 3.2e-2}
TOL_LSE = 1e-3

CASES = [(w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, w.seed) for w in DECODE_WORKLOADS] + [
    (2, 3, 16, 5000, 128, "fp16", 71),   # the most query rows the scratch always holds
    (1, 4, 300, 1000, 64, "bf16", 72),   # two CTA tiles of rows, split keys
    (8, 16, 1000, 1000, 64, "bf16", 73),  # 512 CTAs of rows: no split, scratch unused
]


def _close(a_o, a_l, b_o, b_l, dtype, name):
    eo = (a_o.float() - b_o.float()).abs().max().item()
    fin = torch.isfinite(b_l)
    assert torch.equal(torch.isfinite(a_l), fin), f"{name}: -inf rows differ"
    el = (a_l[fin] - b_l[fin]).abs().max().item() if fin.any() else 0.0
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, f"{name}: max|dO| {eo:.3e}, max|dLSE| {el:.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}".format(*c[:6]))
@pytest.mark.parametrize("mask", ["none", "causal", "causal_bottom_right"])
def test_two_calls_in_a_row_match_workspace_entry(cuda_lib, case, mask):
    B, H, Nq, Nk, d, dtype, seed = case
    inputs = [tuple(t.cuda() for t in make_qkv_kv(B, H, Nq, Nk, d, dtype, seed + i)) for i in (0, 1)]
    outs = [(torch.empty_like(q), torch.empty((B, H, Nq), dtype=torch.float32, device="cuda"))
            for q, _, _ in inputs]
    # two static calls back to back on the same stream, then the references
    for (q, k, v), (o, lse) in zip(inputs, outs):
        cuda_lib.fwd_kv_static(q, k, v, o, lse, mask=mask)
    torch.cuda.synchronize()
    for i, ((q, k, v), (o, lse)) in enumerate(zip(inputs, outs)):
        o_ref, l_ref = cuda_lib.fwd_kv(q, k, v, mask=mask, checked=True)
        _close(o, lse, o_ref, l_ref, dtype, f"call {i + 1}")


@pytest.mark.gpu
def test_oversize_is_rejected(cuda_lib):
    B, H, Nq, Nk, d = 1, 64, 256, 65536, 128
    assert cuda_lib.workspace_bytes(B, H, Nq, Nk, d) > cuda_lib.STATIC_SCRATCH_BYTES
    q = torch.zeros((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H, Nk, d), dtype=torch.bfloat16, device="cuda")
    o, lse = torch.empty_like(q), torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    with pytest.raises(cuda_lib.AttnError) as e:
        cuda_lib.fwd_kv_static(q, k, k, o, lse)
    assert e.value.status == cuda_lib.ATTN_ERR_SCRATCH_TOO_SMALL


@pytest.mark.gpu
def test_no_device_memory_is_taken(cuda_lib):
    """After one warm-up call of each kind (module loading, first use of the scratch),
    further calls, split or not, leave the device's free memory (cudaMemGetInfo) and
    torch's allocated bytes unchanged."""
    cases = [(1, 4, 300, 1000, 64, "bf16", 81),   # split keys: partials in the static scratch
             (8, 16, 1000, 1000, 64, "bf16", 82),  # no split
             (2, 3, 16, 5000, 128, "fp16", 83)]    # split, d = 128
    bufs = []
    for B, H, Nq, Nk, d, dtype, seed in cases:
        q, k, v = (t.cuda() for t in make_qkv_kv(B, H, Nq, Nk, d, dtype, seed))
        bufs.append((q, k, v, torch.empty_like(q), torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")))
    for mask in ("none", "causal_bottom_right"):
        for q, k, v, o, lse in bufs:
            cuda_lib.fwd_kv_static(q, k, v, o, lse, mask=mask)
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for _ in range(3):
        for mask in ("none", "causal_bottom_right"):
            for q, k, v, o, lse in bufs:
                cuda_lib.fwd_kv_static(q, k, v, o, lse, mask=mask)
    torch.cuda.synchronize()
    free1, alloc1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    assert alloc1 == alloc0, f"torch allocated {alloc1 - alloc0} bytes"
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
