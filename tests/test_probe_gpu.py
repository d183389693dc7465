"""One-tile tensor-core probe: checks the TMA maps, the 128-byte-swizzle shared
memory descriptors (K-major and MN-major), the instruction descriptors and the
TMEM load/store layouts that the forward kernel is built from."""
import numpy as np
import pytest
import torch

from gen import make_qkv, to_dtype


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_probe_tile_products(cuda_lib, d, dtype):
    q, k, v = make_qkv(1, 1, 128, d, dtype, seed=500 + d)
    g = torch.Generator().manual_seed(77)
    p = torch.rand((128, 128), generator=g).to(to_dtype(dtype))
    s, o = cuda_lib.probe_tile(q[0, 0].cuda(), k[0, 0].cuda(), v[0, 0].cuda(), p.cuda())
    torch.cuda.synchronize()
    q64, k64, v64, p64 = (t.to(torch.float64).numpy() for t in (q[0, 0], k[0, 0], v[0, 0], p))
    s_ref = q64 @ k64.T
    o_ref = p64 @ v64
    s_err = np.abs(s.cpu().double().numpy() - s_ref).max()
    o_err = np.abs(o.cpu().double().numpy() - o_ref).max()
    # products of 16-bit values are exact in fp32; only the fp32 accumulation rounds
    assert s_err <= 1e-4 * max(1.0, np.abs(s_ref).max()), f"S = QK^T max err {s_err}"
    assert o_err <= 1e-4 * max(1.0, np.abs(o_ref).max()), f"O = PV max err {o_err}"


@pytest.mark.gpu
def test_bounded_wait_times_out_and_the_context_survives(cuda_lib):
    """A wait that nothing completes gives up after the kernels' limit, records where,
    and the other warp stops on the abort flag; a forward afterwards still works."""
    import math
    import time

    import numpy as np
    import torch

    import oracle
    from gen import make_qkv

    t0 = time.perf_counter()
    st = cuda_lib.load().attn_probe_wait_timeout(None)
    dt = time.perf_counter() - t0
    assert st == cuda_lib.ATTN_ERR_TIMEOUT
    assert 1.0 < dt < 10.0
    code, block, where, it = cuda_lib.device_error_info()
    assert (code, block, where, it) == (1, 0, 9000, 7)
    q, k, v = make_qkv(1, 2, 200, 64, "fp16", seed=99)
    o, lse = cuda_lib.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True, checked=True)
    o_ref, _ = oracle.attn_fwd(q, k, v, True, 1.0 / math.sqrt(64))
    assert np.abs(o.double().cpu().numpy() - o_ref).max() <= 4e-3
    assert torch.cuda.synchronize() is None
