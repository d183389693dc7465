"""Host logic of bench.py, on the CPU: throughput aggregation, the max-over-ranks
reduction across two gloo ranks, clock summaries, the ncu-traffic bookkeeping and
the reference (oracle) arm's JSON line, and the L2 flush helper."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_step_flops_and_aggregate():
    f = bench.step_flops()
    assert f == pytest.approx(274.877906944e9 * 1.5)
    a = bench.aggregate([0.4, 0.5], f, world=2)
    assert a["ms_per_step"] == 0.5
    assert a["value"] == pytest.approx(2 * f / 0.5e-3 / 1e12)


def test_defaults_meet_the_timing_rules():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"


def test_clock_summary():
    s = [{"t": 1.0, "sm": 1900, "sm_max": 2070, "power": 900, "reasons": []},
         {"t": 2.0, "sm": 1800, "sm_max": 2070, "power": 1300, "reasons": ["sw_power_cap"]},
         {"t": 3.0, "sm": 2000, "sm_max": 2070, "power": 1000, "reasons": []},
         {"t": 9.0, "sm": 300, "sm_max": 2070, "power": 90, "reasons": []}]
    c = bench.summarize_clocks(s, 0.5, 3.5)
    assert c["sm_mhz"] == 1900 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3


def test_traffic_only_for_the_profiled_kernel(tmp_path):
    p = tmp_path / "summary.md"
    p.write_text(f"kernel_source_sha256: {bench.kernel_source_hash()}\n"
                 "dram_bytes_per_launch_noncausal: 123456\n")
    assert bench.profiled_traffic(str(p)) == 123456
    p.write_text("kernel_source_sha256: 0000000000000000\ndram_bytes_per_launch_noncausal: 1\n")
    assert bench.profiled_traffic(str(p)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md")) is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = bench.allreduce_max([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)], world)
    agg = bench.aggregate([vals[0]], 1e12, world)
    q.put((rank, vals, agg))
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, vals, agg in out:
        assert vals == [2.0, 5.0, 0.5]            # element-wise max over both ranks
        assert agg["value"] == pytest.approx(2e12 / 2e-3 / 1e12)  # both ranks' work / slowest time


def _run_bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_json_line():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0",
                    "--ref-step-seconds", "0.2"])
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in j
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == "TFLOP/s"
    assert j["value"] > 0 and j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["value"] == j["value"]


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_decode_bytes():
    import bench
    # b8h32q1k8192d128 bf16: K and V dominate; Q, O and LSE add a little
    kv = 2 * 8 * 32 * 8192 * 128 * 2
    qo = 2 * 8 * 32 * 1 * 128 * 2
    assert bench.decode_bytes(8, 32, 1, 8192, 128) == kv + qo + 4 * 8 * 32
    from gen import DECODE_WORKLOADS, decode_workload
    for w in DECODE_WORKLOADS:
        assert decode_workload(w.name) is w
    assert bench.parse_args(["--decode", "b8h32q1k8192d128"]).decode == "b8h32q1k8192d128"


def test_bwd_flops():
    import bench
    from exact_attention_61_gb300 import counts
    # five N x N x d products against the forward's two
    assert bench.bwd_flops(4, 16, 4096, 64, False) == 2.5 * counts.attn_flops(4, 16, 4096, 64, False)
    assert bench.bwd_flops(4, 16, 4096, 64, True) == 2.5 * counts.attn_flops(4, 16, 4096, 64, True)
    assert bench.parse_args(["--bwd"]).bwd


def test_fwd_bytes_and_exps():
    # q, k, v, o: 4 tensors of B*H*N*d bf16; lse: B*H*N fp32
    assert bench.fwd_bytes(4, 16, 4096, 64) == 4 * 2 * 4 * 16 * 4096 * 64 + 4 * 4 * 16 * 4096
    assert bench.softmax_exps(1, 1, 4, False) == 16
    assert bench.softmax_exps(1, 1, 4, True) == 10          # 1 + 2 + 3 + 4 unmasked scores
    assert bench.softmax_exps(2, 3, 5, True) == 6 * 15
    assert bench.ex2_peak(152, 2000.0) == pytest.approx(32 * 152 * 2e9)
    for b_, h_, n_, d_, causal in bench.HBM_SWEEP:
        assert b_ * n_ == 16384 and h_ == 16 and d_ == 64


def test_cpu_model_parsing():
    x86 = "processor\t: 0\nvendor_id\t: GenuineIntel\nmodel name\t: Intel(R) Xeon(R) Platinum 8480+\n"
    assert bench.cpu_model(x86) == "Intel(R) Xeon(R) Platinum 8480+"
    arm = "processor\t: 0\nBogoMIPS\t: 2000.00\nCPU implementer\t: 0x41\nCPU architecture: 8\nCPU part\t: 0xd4f\n"
    assert bench.cpu_model(arm).startswith("Arm Neoverse-V2")
    odd = "CPU implementer\t: 0x61\nCPU part\t: 0x022\n"
    assert bench.cpu_model(odd) == "Arm implementer 0x61, part 0x022"
    assert bench.cpu_model("") == "unknown"
    assert isinstance(bench.cpu_model(), str)


def test_spot_check_flags_errors():
    import numpy as np
    rng = np.random.default_rng(0)
    o_ref, l_ref = rng.standard_normal((8, 64)), rng.standard_normal(8)
    r = bench.spot_check(o_ref + 0.01, l_ref + 1e-4, o_ref, l_ref)
    assert r["ok"] and r["rows"] == 8 and r["over_tol_o"] == 0
    bad = o_ref.copy()
    bad[3, 5] += 0.05
    r = bench.spot_check(bad, l_ref, o_ref, l_ref)
    assert not r["ok"] and r["over_tol_o"] == 1 and r["max_abs_err_o"] == pytest.approx(0.05)
    r = bench.spot_check(o_ref, l_ref + 2e-3, o_ref, l_ref)
    assert not r["ok"] and r["over_tol_lse"] == 8


def test_l2_flush_writes_then_reads_without_a_copy():
    """The flush writes a buffer of twice the L2 size (64 MB at least), then sums a float32
    buffer of the same size: float32 sums in place, with no widening copy (an int32 buffer
    would first be copied to int64, a second large write)."""
    import torch
    calls = []

    class Spy(torch.Tensor):
        pass

    f = bench.L2Flush(torch, "cpu", 1 << 20)
    n = 2 * (64 << 20)
    assert f.w.numel() == n and f.w.dtype == torch.uint8
    assert f.r.numel() * f.r.element_size() == n and f.r.dtype == torch.float32
    assert f.r.sum().dtype == torch.float32  # no promotion, so no widening copy
    orig = f.r
    f.r = orig.as_subclass(Spy)
    torch_sum = Spy.sum

    def spy_sum(self, *a, **k):
        calls.append(1)
        return torch_sum(self, *a, **k)

    Spy.sum = spy_sum
    f(7)
    assert int(f.w[0]) == 7 and int(f.w[-1]) == 7 and calls == [1]
    f(8, write_only=True)
    assert int(f.w[0]) == 8 and calls == [1]
