"""attn_fwd_host (inputs and outputs in host memory, copies pipelined with the kernels by
chunks of heads) through the C ABI: parity with the fp64 oracle on small problems, and
bit-for-bit equality with the device-memory path (attn_fwd, the same kernel on the same
heads) at sizes that make several chunks, with page-locked and pageable host buffers and
with work before and after the call on the caller's stream."""
import math
import threading

import numpy as np
import pytest
import torch

import oracle
from gen import make_qkv

TOL_O = {"fp16": 4e-3, "bf16": 3.2e-2}
TOL_LSE = 1e-3


def _device_ref(attn, q, k, v, causal, scale):
    o, lse = attn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, checked=True)
    return o.cpu(), lse.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,d,dtype", [(1, 3, 300, 64, "bf16"), (2, 2, 129, 128, "fp16"),
                                           (1, 1, 1, 64, "fp16"), (1, 2, 513, 128, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
def test_small_matches_oracle(cuda_lib, B, H, N, d, dtype, causal):
    q, k, v = make_qkv(B, H, N, d, dtype, 66000 + N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = cuda_lib.fwd_host(q, k, v, causal=causal, scale=scale, checked=True)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    eo = np.abs(o.to(torch.float64).numpy() - o_ref).max()
    el = np.abs(lse.to(torch.float64).numpy() - lse_ref).max()
    assert eo <= TOL_O[dtype] and el <= TOL_LSE, (eo, el)
    od, ld = _device_ref(cuda_lib, q, k, v, causal, scale)
    assert torch.equal(o, od) and torch.equal(lse, ld)


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_headline_size_in_chunks_equals_device_path(cuda_lib, causal):
    """B=4, H=16, N=4096, d=64, bf16: four chunks (19, 19, 19, 7 heads)."""
    B, H, N, d = 4, 16, 4096, 64
    assert cuda_lib.host_plan(B, H, N, d) == (4, 19)
    q, k, v = make_qkv(B, H, N, d, "bf16", 66100 + int(causal))
    scale = 1.0 / math.sqrt(d)
    o, lse = cuda_lib.fwd_host(q, k, v, causal=causal, scale=scale, checked=True)
    od, ld = _device_ref(cuda_lib, q, k, v, causal, scale)
    assert torch.equal(o, od) and torch.equal(lse, ld)
    # a few rows of each chunk against the oracle, computed one by one
    rows = np.array([h * N + r for h in (0, 18, 19, 38, 57, 63) for r in (0, 1, 2047, N - 1)], dtype=np.int64)
    o_ref, lse_ref = oracle.attn_fwd_rows(q, k, v, causal, rows, scale)
    og = o.reshape(-1, d)[torch.from_numpy(rows)].to(torch.float64).numpy()
    lg = lse.reshape(-1)[torch.from_numpy(rows)].to(torch.float64).numpy()
    assert np.abs(og - o_ref).max() <= TOL_O["bf16"] and np.abs(lg - lse_ref).max() <= TOL_LSE


@pytest.mark.gpu
def test_pageable_buffers_and_a_reused_workspace(cuda_lib):
    B, H, N, d = 2, 20, 2048, 128  # 2 chunks: 38 and 2 heads
    assert cuda_lib.host_plan(B, H, N, d) == (2, 38)
    ws = torch.empty((cuda_lib.host_workspace_bytes(B, H, N, d),), dtype=torch.uint8, device="cuda")
    o = torch.empty((B, H, N, d), dtype=torch.float16)   # pageable
    lse = torch.empty((B, H, N), dtype=torch.float32)    # pageable
    for seed, causal in ((66200, False), (66201, True)):
        q, k, v = make_qkv(B, H, N, d, "fp16", seed)
        cuda_lib.fwd_host(q, k, v, causal=causal, out=o, lse=lse, workspace=ws, checked=True)
        od, ld = _device_ref(cuda_lib, q, k, v, causal, 1.0 / math.sqrt(d))
        assert torch.equal(o, od) and torch.equal(lse, ld)


@pytest.mark.gpu
def test_ordered_with_work_on_the_callers_stream(cuda_lib):
    """On a side stream: a device-to-host copy writes the host inputs, then attn_fwd_host
    reads them, then a host-to-device copy reads its host outputs. With the copies ordered
    by the stream, the inputs are the new ones and the outputs read back are complete."""
    B, H, N, d = 8, 16, 1024, 64  # 2 chunks: 76 and 52 heads
    assert cuda_lib.host_plan(B, H, N, d) == (2, 76)
    q0, k, v = make_qkv(B, H, N, d, "bf16", 66300)
    q1 = make_qkv(B, H, N, d, "bf16", 66301)[0]
    qh = q0.clone().pin_memory()
    kh, vh = k.pin_memory(), v.pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    lh = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty((cuda_lib.host_workspace_bytes(B, H, N, d),), dtype=torch.uint8, device="cuda")
    q1d = q1.cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)       # keep the stream busy so that ordering matters
        qh.copy_(q1d, non_blocking=True)   # new inputs arrive through the stream
        st = cuda_lib.attn_fwd_host(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), lh.data_ptr(),
                                    B, H, N, d, True, 0.125, cuda_lib.ATTN_BF16, ws.data_ptr(), ws.numel(),
                                    s.cuda_stream)
        assert st == cuda_lib.ATTN_OK
        back = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
        back.copy_(oh, non_blocking=True)  # reads the host output after the call
    s.synchronize()
    od, ld = _device_ref(cuda_lib, q1, k, v, True, 0.125)
    assert torch.equal(oh, od) and torch.equal(lh, ld)
    assert torch.equal(back.cpu(), od)


@pytest.mark.gpu
def test_two_host_threads_on_two_streams(cuda_lib):
    B, H, N, d = 8, 16, 1024, 64  # 2 chunks each
    cases = [make_qkv(B, H, N, d, "bf16", 66400 + i) for i in range(2)]
    out = [None, None]
    errs = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(3):
                    out[i] = cuda_lib.fwd_host(*cases[i], causal=bool(i), stream=s)
        except Exception as e:  # reported below
            errs.append(e)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    for i in range(2):
        od, ld = _device_ref(cuda_lib, *cases[i], bool(i), 0.125)
        assert torch.equal(out[i][0], od) and torch.equal(out[i][1], ld)


@pytest.mark.gpu
def test_second_mask_on_the_staged_inputs(cuda_lib):
    """The second call passes q = k = v = NULL and reuses what the first staged."""
    B, H, N, d = 4, 16, 2048, 64  # 2 chunks
    q, k, v = make_qkv(B, H, N, d, "bf16", 66500)
    ws = torch.empty((cuda_lib.host_workspace_bytes(B, H, N, d),), dtype=torch.uint8, device="cuda")
    outs = []
    for causal in (False, True):
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory()
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        ins = (q, k, v) if not causal else (None, None, None)
        outs.append(cuda_lib.fwd_host(*ins, causal=causal, out=o, lse=lse, workspace=ws, checked=True))
    for causal, (o, lse) in zip((False, True), outs):
        od, ld = _device_ref(cuda_lib, q, k, v, causal, 0.125)
        assert torch.equal(o, od) and torch.equal(lse, ld)
