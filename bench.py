"""Benchmark of the fused attention forward on GB300.

One step = one pass of the whole hot path over the B=4, H=16, N=4096, d=64 bf16
problem: the non-causal forward and the causal forward (causal tile skipping is
part of the path), each one launch of the sm_103a kernel through the C ABI.
FLOPs per step = 4*B*H*N^2*d + (4*B*H*N^2*d)/2 (the causal half), the
convention of the profile-driven FlashAttention-2 page (Round 0 / Step 5).

Timing: W warm-up steps (plus enough extra steps to keep the GPU busy for
--warmup-seconds, so clocks have ramped), peak-memory counters reset after
warm-up, then K steps timed with CUDA events on the launching stream, the L2
cache flushed before every step outside the events (a write of twice its size,
then a read of another buffer of twice its size, so that the write's dirty lines
go back to HBM before the step rather than inside it), a barrier and a synchronize on both sides of the timed region, max over ranks.
`value`, `ms_per_step` and `roofline.achieved` come from the per-step medians
(the means, p10 and p90 are reported beside them).

After the timed region, outside it: a second pass of K flushed steps (the run
repeated, to show its spread), K steps without the L2 flush, the HBM-bound
points of the sequence sweep, and the end-to-end call from host buffers. The
cpu_baseline leg times the fp64 oracle on sampled rows and compares those rows
with the outputs of the last timed launch of each mask.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0. With --gpus N > 1 (under torchrun) every rank
runs an independent replica of the same problem on its own GPU; nothing is
exchanged on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s at B=4,H=16,N=4096,d=64 bf16; % of tensor-core peak"
UNIT = "TFLOP/s"
B, H, N, D = 4, 16, 4096, 64
DTYPE = "bf16"
SEED = 61002
WORKLOAD = "b4h16n4096d64 bf16, non-causal + causal forward per step"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attn_fwd_b4h16n4096d64.md")
KERNEL_SOURCES = ["exact_attention_61_gb300/csrc/attn_fwd_persist.cuh",
                  "exact_attention_61_gb300/csrc/attn_fwd_kernel.cuh",
                  "exact_attention_61_gb300/csrc/sm103_ptx.cuh",
                  "exact_attention_61_gb300/csrc/attn_internal.h",
                  "exact_attention_61_gb300/csrc/attn_fwd_inst.cu"]


# The sequence-sweep points that are bound by HBM rather than by the tensor cores
# (B = 16384 / N, H = 16, d = 64): short rows leave little compute per byte moved.
HBM_SWEEP = [(32, 16, 512, 64, False), (32, 16, 512, 64, True), (16, 16, 1024, 64, True)]
# Tolerances of the parity check (bf16 O, and the LSE in natural-log units).
TOL_O, TOL_LSE = 3.2e-2, 1e-3
# ex2 results per SM per clock: 16 on sm_100 parts, doubled on Blackwell Ultra (sm_103).
EX2_PER_SM_CLK = 32


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------------------------
# pure host logic (tested on the CPU)
# ---------------------------------------------------------------------------------------------

def step_flops() -> float:
    from exact_attention_61_gb300 import counts
    return counts.attn_flops(B, H, N, D, False) + counts.attn_flops(B, H, N, D, True)


def tflops(flops: float, ms: float) -> float:
    return flops / (ms * 1e-3) / 1e12


def fwd_bytes(B_: int, H_: int, N_: int, d: int, elem: int = 2) -> int:
    """Algorithmic HBM bytes of one forward: q, k, v read once, o and the fp32 LSE
    written once."""
    return 4 * elem * B_ * H_ * N_ * d + 4 * B_ * H_ * N_


def softmax_exps(B_: int, H_: int, N_: int, causal: bool) -> int:
    """Exponentials the softmax takes by definition: one per unmasked score."""
    per_head = N_ * (N_ + 1) // 2 if causal else N_ * N_
    return B_ * H_ * per_head


def ex2_peak(sms: int, sm_mhz: float) -> float:
    """Nominal ex2 throughput (results/s) of `sms` SMs at `sm_mhz`."""
    return EX2_PER_SM_CLK * sms * sm_mhz * 1e6


def cpu_model(cpuinfo: str | None = None) -> str:
    """The host CPU's model from /proc/cpuinfo: the x86 'model name' line, else the
    Arm implementer and part numbers (named where known)."""
    if cpuinfo is None:
        try:
            with open("/proc/cpuinfo") as f:
                cpuinfo = f.read()
        except OSError:
            return "unknown"
    fields = {}
    for line in cpuinfo.splitlines():
        if ":" in line:
            key, val = line.split(":", 1)
            fields.setdefault(key.strip().lower(), val.strip())
    if fields.get("model name"):
        return fields["model name"]
    impl, part = fields.get("cpu implementer"), fields.get("cpu part")
    if impl and part:
        known = {("0x41", "0xd4f"): "Arm Neoverse-V2", ("0x41", "0xd40"): "Arm Neoverse-V1",
                 ("0x41", "0xd0c"): "Arm Neoverse-N1", ("0x41", "0xd8e"): "Arm Neoverse-N3",
                 ("0x41", "0xd84"): "Arm Neoverse-V3"}
        name = known.get((impl.lower(), part.lower()))
        return f"{name} (implementer {impl}, part {part})" if name else f"Arm implementer {impl}, part {part}"
    return "unknown"


def spot_check(o_gpu, lse_gpu, o_ref, lse_ref, tol_o: float = TOL_O, tol_lse: float = TOL_LSE) -> dict:
    """Element-wise comparison of sampled output rows (numpy arrays, [R, d] and [R])."""
    import numpy as np
    d_o = np.abs(np.asarray(o_gpu, dtype=np.float64) - o_ref)
    d_l = np.abs(np.asarray(lse_gpu, dtype=np.float64) - lse_ref)
    return {"rows": int(d_l.size), "max_abs_err_o": float(d_o.max(initial=0.0)),
            "max_abs_err_lse": float(d_l.max(initial=0.0)),
            "over_tol_o": int((d_o > tol_o).sum()), "over_tol_lse": int((d_l > tol_lse).sum()),
            "tol_o": tol_o, "tol_lse": tol_lse,
            "ok": bool((d_o <= tol_o).all() and (d_l <= tol_lse).all())}


def aggregate(ms_per_rank, flops_per_rank_step: float, world: int) -> dict:
    """Whole-job throughput: all ranks' work over the slowest rank's time."""
    ms = max(ms_per_rank)
    return {"ms_per_step": ms, "value": tflops(flops_per_rank_step * world, ms)}


def allreduce_max(values, world: int, device=None):
    """Element-wise maximum of `values` over all ranks (identity for one rank)."""
    if world <= 1:
        return [float(x) for x in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x) for x in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_path: str = PROFILE_SUMMARY):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    or None if there is none or the kernel source changed since it was taken."""
    if not os.path.exists(summary_path):
        return None
    text = open(summary_path).read()
    mh = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    mt = re.search(r"dram_bytes_per_launch_noncausal:\s*([0-9]+)", text)
    if not mh or not mt or mh.group(1) != kernel_source_hash():
        return None
    return int(mt.group(1))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return {"bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "hbm_gbs": float(j.get("hbm_gbs", 6800.0)), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def summarize_clocks(samples, t0: float, t1: float) -> dict:
    """Median SM clock and active throttle reasons over samples taken in [t0, t1]."""
    win = [s for s in samples if t0 <= s["t"] <= t1]
    if not win:
        win = samples[-3:]
    if not win:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    reasons = sorted({r for s in win for r in s["reasons"]})
    return {"sm_mhz": statistics.median(s["sm"] for s in win),
            "sm_max_mhz": max(s["sm_max"] for s in win),
            "power_w_max": max(s["power"] for s in win),
            "reasons": reasons, "samples": len(win)}


class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.samples = []
        self.error = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={','.join(self.FIELDS)}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.proc = None
            self.error = str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                self.samples.append({
                    "t": time.time(), "sm": float(parts[0]), "sm_max": float(parts[1]),
                    "power": float(parts[2]) if parts[2] not in ("[N/A]", "N/A") else 0.0,
                    "reasons": [r for r, v in zip(self.REASONS, parts[3:]) if v == "Active"]})
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()


# ---------------------------------------------------------------------------------------------
# CPU baseline: the fp64 oracle on the host cores, on a bounded sample of the workload
# ---------------------------------------------------------------------------------------------

def _sample_rows(n_rows: int, seed: int = 0):
    import numpy as np
    rng = np.random.default_rng(seed)
    return rng.integers(0, B * H * N, size=n_rows).astype(np.int64)


def _row_flops(rows, causal: bool) -> float:
    if not causal:
        return 4.0 * N * D * len(rows)
    return float(sum(4.0 * ((int(r) % N) + 1) * D for r in rows))


def oracle_rate(q64, k64, v64, n_rows: int, seed: int = 0, keep: bool = False):
    """Time the oracle on n_rows sampled query rows under each mask. Returns
    (FLOPs, seconds), and with keep=True also (rows, {causal: (O rows, LSE rows)})."""
    import oracle
    rows = _sample_rows(n_rows, seed)
    scale = 1.0 / math.sqrt(D)
    flops = secs = 0.0
    outs = {}
    for causal in (False, True):
        t0 = time.perf_counter()
        outs[causal] = oracle.attn_fwd_rows(q64, k64, v64, causal, rows, scale)
        secs += time.perf_counter() - t0
        flops += _row_flops(rows, causal)
    if keep:
        return flops, secs, rows, outs
    return flops, secs


def calibrate_rows(q64, k64, v64, target_s: float) -> int:
    n = 64
    while True:
        _, s = oracle_rate(q64, k64, v64, n, seed=1)
        if s >= 0.5 or n >= 1 << 20:
            return max(16, int(n * target_s / max(s, 1e-6)))
        n *= 4


def cpu_baseline(q, k, v, target_s: float = 12.0, timed_outputs=None) -> dict:
    """The fp64 oracle on the host cores over a bounded sample of rows. With
    `timed_outputs` = {causal: (O [B,H,N,d], LSE [B,H,N]) on the host}, the sampled rows
    are also compared with those outputs of the timed launches."""
    import oracle
    q64, k64, v64 = oracle.to_f64(q), oracle.to_f64(k), oracle.to_f64(v)
    n = calibrate_rows(q64, k64, v64, target_s)
    flops, secs, rows, outs = oracle_rate(q64, k64, v64, n, seed=2, keep=True)
    res = {"value": tflops(flops, secs * 1e3), "unit": UNIT, "cores": oracle.num_threads(),
           "cpu_model": cpu_model(), "kind": "oracle",
           "sample": f"{n} random query rows of the B=4,H=16,N=4096,d=64 bf16 problem, "
                     f"each under both masks, fp64 C oracle; {secs:.1f} s of CPU work"}
    if timed_outputs is not None:
        res["parity_of_timed_outputs"] = {}
        import torch
        idx = torch.from_numpy(rows)
        for causal, (o_h, l_h) in timed_outputs.items():
            o_rows = o_h.reshape(-1, D)[idx].double().numpy()
            l_rows = l_h.reshape(-1)[idx].double().numpy()
            res["parity_of_timed_outputs"]["causal" if causal else "noncausal"] = spot_check(
                o_rows, l_rows, outs[causal][0], outs[causal][1])
    return res


# ---------------------------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------------------------

def rank_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


L2_NOTE = ("flushed before every step outside the events: a write of 2x L2 size, then a read of "
           "another 2x L2 buffer that writes the dirty lines back before the step")


class L2Flush:
    """Evicts a step's inputs from L2 between steps, outside the timed region.

    A write of twice the L2 size evicts every input line but leaves L2 full of dirty
    lines, which the next step would then write back to HBM inside its own timed
    region (about 126 MB: 9-12 % of an HBM-bound decode step). A read of a second
    buffer of twice the L2 size afterwards writes them back first, so the step starts
    from a cold, clean L2 as the first step after a read-only phase would.
    ``write_only=True`` keeps the bare write, for the comparison figure."""

    def __init__(self, torch, dev, l2: int):
        n = 2 * max(l2, 64 << 20)
        self.w = torch.empty(n, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(n // 4, dtype=torch.float32, device=dev)  # summed in place, no copy

    def __call__(self, i: int, write_only: bool = False):
        self.w.fill_(i & 0xFF)
        if not write_only:
            self.r.sum()


def run_reference(args) -> int:
    rank, _, world = rank_env()
    if rank != 0:
        return 0
    import oracle
    from gen import make_qkv
    q, k, v = make_qkv(B, H, N, D, DTYPE, SEED)
    q64, k64, v64 = oracle.to_f64(q), oracle.to_f64(k), oracle.to_f64(v)
    n = calibrate_rows(q64, k64, v64, target_s=args.ref_step_seconds)
    for i in range(max(args.warmup, 0)):
        oracle_rate(q64, k64, v64, n, seed=100 + i)
    total_f = total_s = 0.0
    for i in range(args.steps):
        f, s = oracle_rate(q64, k64, v64, n, seed=1000 + i)
        total_f += f
        total_s += s
    value = tflops(total_f, total_s * 1e3)
    ms = total_s * 1e3 / max(args.steps, 1)
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic",
           "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D,
                      "step": f"{n} sampled query rows x both masks"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                            "cpu_model": cpu_model(), "kind": "oracle",
                            "sample": f"{n} random query rows per step under both masks, fp64 C oracle"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def run_ours(args) -> int:
    import torch
    import torch.distributed as dist

    from exact_attention_61_gb300 import attn, counts
    from gen import make_qkv

    rank, local_rank, world = rank_env()
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device for --impl ours")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    attn.load()

    def barrier():
        if world > 1:
            dist.barrier()

    q_h, k_h, v_h = make_qkv(B, H, N, D, DTYPE, SEED)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    # one output pair per mask, so that both timed launches' outputs survive the step
    o = {c: torch.empty_like(q) for c in (False, True)}
    lse = {c: torch.empty((B, H, N), dtype=torch.float32, device=dev) for c in (False, True)}
    scale = 1.0 / math.sqrt(D)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = L2Flush(torch, dev, l2)
    dt = attn.ATTN_BF16

    def launch(causal, q_=q, k_=k, v_=v, o_=None, l_=None, shape=(B, H, N, D)):
        o_ = o[causal] if o_ is None else o_
        l_ = lse[causal] if l_ is None else l_
        st = attn.attn_fwd(q_.data_ptr(), k_.data_ptr(), v_.data_ptr(), o_.data_ptr(), l_.data_ptr(),
                           *shape, causal, 1.0 / math.sqrt(shape[3]), dt, sptr)
        if st != attn.ATTN_OK:
            raise RuntimeError(f"attn_fwd failed: {attn.strerror(st)}")

    def timed_steps(n, flush_l2=True):
        """n steps (non-causal then causal launch), per-launch CUDA-event times in ms."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        for i in range(n):
            if flush_l2:
                flush(i)
            ev[i][0].record(stream)
            launch(False)
            ev[i][1].record(stream)
            launch(True)
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
        return ([ev[i][0].elapsed_time(ev[i][1]) for i in range(n)],
                [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)])

    sampler = ClockSampler(local_rank) if args.clocks else None
    # ---- warm-up: W steps, then keep the GPU busy until --warmup-seconds have passed -----
    t_w = time.perf_counter()
    n_warm = 0
    while n_warm < args.warmup or time.perf_counter() - t_w < args.warmup_seconds:
        flush(n_warm)
        launch(False)
        launch(True)
        n_warm += 1
        if n_warm % 16 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)

    # ---- timed region: exactly K steps --------------------------------------------------
    barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    w0 = time.perf_counter()
    t_nc, t_c = timed_steps(args.steps)
    barrier()
    wall_s = time.perf_counter() - w0
    t1 = time.time()
    launches = 2 * args.steps
    t_step = [a + b for a, b in zip(t_nc, t_c)]
    peak_mem_gb = torch.cuda.max_memory_allocated(dev) / 1e9
    # outputs of the last timed launch of each mask, for the parity spot check
    timed_out = {c: (o[c].cpu(), lse[c].cpu()) for c in (False, True)}

    # ---- outside the timed region: the run repeated, and the same steps without the flush --
    r_nc, r_c = timed_steps(args.steps)
    n_nc, n_c = timed_steps(args.steps, flush_l2=False)
    t2 = time.time()

    # ---- the HBM-bound points of the sequence sweep (flushed, outside the timed region) ---
    sweep = []
    peaks = measured_peaks()
    for (b_, h_, n_, d_, causal) in HBM_SWEEP:
        qs, ks, vs = (t.to(dev) for t in make_qkv(b_, h_, n_, d_, DTYPE, SEED + 7))
        os_, ls_ = torch.empty_like(qs), torch.empty((b_, h_, n_), dtype=torch.float32, device=dev)
        ts = []
        for i in range(max(3, args.warmup) + args.steps):
            flush(i)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch(causal, qs, ks, vs, os_, ls_, (b_, h_, n_, d_))
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize(dev)
        ms_s = statistics.median(a.elapsed_time(b) for a, b in ts[max(3, args.warmup):])
        by = fwd_bytes(b_, h_, n_, d_)
        sweep.append({"B": b_, "H": h_, "N": n_, "d": d_, "causal": causal, "ms_median": ms_s,
                      "tflops": tflops(counts.attn_flops(b_, h_, n_, d_, causal), ms_s),
                      "algorithmic_bytes": by, "gbs": by / (ms_s * 1e-3) / 1e9,
                      "hbm_frac": by / (ms_s * 1e-3) / 1e9 / peaks["hbm_gbs"]})
        del qs, ks, vs, os_, ls_

    # ---- end to end through the C ABI with host buffers (copies inside the timed region) --
    # attn_fwd_host, once per mask: the first call copies q, k, v from page-locked host
    # memory into the workspace, the second reuses them there (q = k = v = NULL); each runs
    # the forward and copies its o, lse back, pipelined by chunks of heads.
    qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
    o_host = [torch.empty_like(qp).pin_memory() for _ in range(2)]
    l_host = [torch.empty((B, H, N), dtype=torch.float32).pin_memory() for _ in range(2)]
    ws = torch.empty((attn.host_workspace_bytes(B, H, N, D),), dtype=torch.uint8, device=dev)
    n_chunks, heads_per_chunk = attn.host_plan(B, H, N, D)
    e2e_steps = max(3, min(args.steps, 50))
    h2d = 3 * q_h.numel() * q_h.element_size()
    d2h = 2 * (q.numel() * q.element_size() + B * H * N * 4)

    def e2e_step():
        for j, causal in enumerate((False, True)):
            ins = (qp.data_ptr(), kp.data_ptr(), vp.data_ptr()) if j == 0 else (None, None, None)
            st = attn.attn_fwd_host(*ins, o_host[j].data_ptr(), l_host[j].data_ptr(), B, H, N, D, causal, scale,
                                    dt, ws.data_ptr(), ws.numel(), sptr)
            if st != attn.ATTN_OK:
                raise RuntimeError(f"attn_fwd_host failed: {attn.strerror(st)}")

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms_local = e_start.elapsed_time(e_end) / e2e_steps
    if sampler:
        sampler.stop()

    # ---- aggregate over ranks (medians per rank, max over ranks) ---------------------------
    med = statistics.median
    ms, e2e_ms, ms_nc, ms_c = allreduce_max([med(t_step), e2e_ms_local, med(t_nc), med(t_c)], world, dev)
    if rank == 0:
        f_nc = counts.attn_flops(B, H, N, D, False)
        f_c = counts.attn_flops(B, H, N, D, True)
        agg = aggregate([ms], f_nc + f_c, world)
        achieved = tflops(f_nc, ms_nc)
        traffic = profiled_traffic()
        clocks = summarize_clocks(sampler.samples, t0 - args.warmup_seconds, t1) if sampler else None
        sm_mhz = (clocks or {}).get("sm_mhz") or 0.0

        def kstats(ts, f, causal):
            m = med(ts)
            e = softmax_exps(B, H, N, causal)
            r = {"ms_median": m, "ms_mean": statistics.fmean(ts), "ms_p10": _pct(ts, 10),
                 "ms_p90": _pct(ts, 90), "tflops": tflops(f, m),
                 "frac_of_peak": tflops(f, m) / peaks["bf16_tflops"],
                 "exps_per_s": e / (m * 1e-3)}
            if sm_mhz:
                r["exps_frac_of_ex2_peak"] = r["exps_per_s"] / ex2_peak(sms, sm_mhz)
            return r

        def pass_summary(a_nc, a_c):
            m_step = med([x + y for x, y in zip(a_nc, a_c)])
            return {"ms_per_step_median": m_step, "tflops": tflops(f_nc + f_c, m_step),
                    "noncausal_tflops": tflops(f_nc, med(a_nc)), "causal_tflops": tflops(f_c, med(a_c))}

        rep_pass = pass_summary(r_nc, r_c)
        rep_pass["diff_vs_timed_pct"] = 100.0 * (rep_pass["ms_per_step_median"] / ms - 1.0)
        nf_pass = pass_summary(n_nc, n_c)
        out = {
            "metric": METRIC, "value": agg["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": n_warm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": B, "H": H, "N": N, "d": D, "scale": scale,
                       "causal": [False, True], "seed": SEED,
                       "l2": L2_NOTE,
                       "statistic": "median over the timed steps (mean, p10, p90 in per_kernel)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "per_kernel": {
                "noncausal": kstats(t_nc, f_nc, False),
                "causal": {**kstats(t_c, f_c, True),
                           "executed_tflops": tflops(counts.kernel_executed_flops(B, H, N, D, True), med(t_c))}},
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_persist_kernel<non-causal, bf16>",
                         "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                         "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"
                         if peaks["source"] == "measured" else "fallback 1.9 PFLOP/s bf16",
                         "algorithmic_flops_per_launch": f_nc,
                         "statistic": "median launch time of the timed steps"},
            "softmax_exps": {"per_step": softmax_exps(B, H, N, False) + softmax_exps(B, H, N, True),
                             "per_s": (softmax_exps(B, H, N, False) + softmax_exps(B, H, N, True)) / (ms * 1e-3),
                             "ex2_peak_per_s": ex2_peak(sms, sm_mhz) if sm_mhz else None,
                             "ex2_peak_basis": f"{EX2_PER_SM_CLK} ex2/clk/SM x {sms} SMs x median SM clock"},
            "repeat": rep_pass,
            "no_l2_flush": {**nf_pass, "note": "the same K steps back to back, L2 not flushed"},
            "hbm_sweep": {"points": sweep, "peak_gbs": peaks["hbm_gbs"],
                          "note": "the HBM-bound points of the sequence sweep (B=16384/N, H=16, d=64), "
                                  "algorithmic bytes (q,k,v read, o,lse written once) / median time"},
            "e2e": {"value": tflops((f_nc + f_c) * world, e2e_ms), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "call": f"attn_fwd_host per mask, the second on the inputs the first staged "
                            f"(page-locked host buffers; copies and kernels pipelined over {n_chunks} "
                            f"chunks of {heads_per_chunk} heads)"},
            "gpu_launches": launches,
            "wall_s_timed_region": wall_s,
            "wall_s_after_timed_region": t2 - t1,
            "peak_mem_gb": peak_mem_gb,
        }
        if clocks is not None:
            out["clocks"] = clocks
        if args.cpu_baseline and world == 1:
            log("timing the fp64 oracle on the host cores ...")
            out["cpu_baseline"] = cpu_baseline(q_h, k_h, v_h, target_s=args.cpu_seconds,
                                               timed_outputs=timed_out)
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def decode_bytes(B_: int, H_: int, Nq: int, Nk: int, d: int, elem: int = 2) -> int:
    """Algorithmic HBM bytes of one decode step: Q, K and V read once, O and the fp32
    LSE written once (the split partials are the implementation's own traffic)."""
    return elem * B_ * H_ * d * (2 * Nq + 2 * Nk) + 4 * B_ * H_ * Nq


def run_decode(args) -> int:
    """--decode NAME: one KV-cache decode step per timed step (attn_fwd_kv, bottom-right
    causal mask: the streaming decode kernel over key ranges, then the merge), reported as
    HBM GB/s against the measured copy bandwidth. Single GPU; an extra measurement beside
    the headline line."""
    import torch

    from exact_attention_61_gb300 import attn
    from gen import decode_workload, make_qkv_kv

    w = decode_workload(args.decode)
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    attn.load()
    q, k, v = (t.to(dev) for t in make_qkv_kv(w.B, w.H, w.Nq, w.Nk, w.d, w.dtype, w.seed))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    ws_n = attn.workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = 1.0 / math.sqrt(w.d)
    dt = attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_FP16
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(torch, dev, l2)

    def launch():
        st = attn.attn_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                              w.B, w.H, w.Nq, w.Nk, w.d, attn.ATTN_MASK_CAUSAL_BOTTOM_RIGHT, scale, dt,
                              ws.data_ptr(), ws_n, stream.cuda_stream)
        if st != attn.ATTN_OK:
            raise RuntimeError(f"attn_fwd_kv failed: {attn.strerror(st)}")

    sampler = ClockSampler(0) if args.clocks else None
    t_w = time.perf_counter()
    n_warm = 0
    while n_warm < args.warmup or time.perf_counter() - t_w < args.warmup_seconds:
        flush(n_warm)
        launch()
        n_warm += 1
        if n_warm % 16 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    def timed(n, write_only=False):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for i in range(n):
            flush(i, write_only)
            ev[i][0].record(stream)
            launch()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    t0 = time.time()
    t_ms = timed(args.steps)
    t1 = time.time()
    if sampler:
        sampler.stop()
    # outside the timed region: the same steps after a bare write flush (its dirty lines are
    # written back inside each step), and back to back without a flush
    t_wo = timed(args.steps, write_only=True)
    t_nf = []
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        t_nf.append((e0, e1))
    torch.cuda.synchronize(dev)
    t_nf = [a.elapsed_time(b) for a, b in t_nf]
    ms = statistics.median(t_ms)
    nbytes = decode_bytes(w.B, w.H, w.Nq, w.Nk, w.d)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    splits = attn.plan_decode_for(w.B * w.H, w.Nq, w.Nk, w.d, ws_n, sms)[0]  # key ranges per head
    out = {
        "metric": f"decode attention HBM GB/s ({w.name})", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": n_warm, "ms_per_step": ms, "higher_is_better": True,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nk": w.Nk, "d": w.d,
                   "mask": "causal_bottom_right", "key_splits": splits, "seed": w.seed,
                   "l2": L2_NOTE, "statistic": "median over the timed steps"},
        "ms_mean": statistics.fmean(t_ms), "ms_p10": _pct(t_ms, 10), "ms_p90": _pct(t_ms, 90),
        "roofline": {"bound": "hbm", "kernel": "attn_decode_kernel + attn_merge_kernel (one call)",
                     "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None,
                     "algorithmic_bytes_per_step": nbytes,
                     "peak_source": "measured copy (MEASURED_PEAKS.json)"
                     if peaks["source"] == "measured" else "fallback 6.8 TB/s"},
        "gpu_launches": (2 if ws_n else 1) * args.steps,
        "l2_write_flush_only": {"ms_median": statistics.median(t_wo),
                                "gbs": nbytes / (statistics.median(t_wo) * 1e-3) / 1e9,
                                "note": "the same steps after a bare 2x L2 write, whose dirty lines "
                                        "are written back inside each step"},
        "no_l2_flush": {"ms_median": statistics.median(t_nf),
                        "gbs": nbytes / (statistics.median(t_nf) * 1e-3) / 1e9,
                        "note": "the same steps back to back (K and V are larger than L2)"},
    }
    if sampler:
        out["clocks"] = summarize_clocks(sampler.samples, t0 - args.warmup_seconds, t1)
    print(json.dumps(out), flush=True)
    return 0


def bwd_flops(B_: int, H_: int, N_: int, d: int, causal: bool) -> float:
    """Algorithmic FLOPs of the backward: five N x N x d products (S, dP, dV, dK, dQ)
    against the forward's two, i.e. 2.5 x 4 B H N^2 d, halved under the causal mask."""
    f = 10.0 * B_ * H_ * N_ * N_ * d
    return f / 2 if causal else f


def run_bwd(args) -> int:
    """--bwd: one backward pass (prep + main kernel + dQ cast) per timed step on the
    headline problem (or --bwd-shape), non-causal then causal, reported as TFLOP/s against the
    measured bf16 peak. Single GPU; an extra measurement beside the headline line."""
    import torch

    from exact_attention_61_gb300 import attn
    from gen import make_qkv

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    B, H, N, D = (int(x) for x in args.bwd_shape.split(","))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    attn.load()
    q, k, v = (t.to(dev) for t in make_qkv(B, H, N, D, DTYPE, SEED))
    do = make_qkv(B, H, N, D, DTYPE, SEED + 7919)[0].to(dev)
    scale = 1.0 / math.sqrt(D)
    outs = {c: attn.fwd(q, k, v, causal=c, scale=scale, checked=True) for c in (False, True)}
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws_n = attn.bwd_workspace_bytes(B, H, N, D)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(torch, dev, l2)

    def launch(causal):
        o, lse = outs[causal]
        st = attn.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                           do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D,
                           causal, scale, attn.ATTN_BF16, ws.data_ptr(), ws_n, stream.cuda_stream)
        if st != attn.ATTN_OK:
            raise RuntimeError(f"attn_bwd failed: {attn.strerror(st)}")

    sampler = ClockSampler(0) if args.clocks else None
    t_w = time.perf_counter()
    n_warm = 0
    while n_warm < args.warmup or time.perf_counter() - t_w < args.warmup_seconds:
        flush(n_warm)
        launch(False)
        launch(True)
        n_warm += 1
        if n_warm % 16 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t0 = time.time()
    for i in range(args.steps):
        flush(i)
        ev[i][0].record(stream)
        launch(False)
        ev[i][1].record(stream)
        launch(True)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if sampler:
        sampler.stop()
    t_nc = [e[0].elapsed_time(e[1]) for e in ev]
    t_c = [e[1].elapsed_time(e[2]) for e in ev]
    ms_nc, ms_c = statistics.median(t_nc), statistics.median(t_c)
    f_nc, f_c = bwd_flops(B, H, N, D, False), bwd_flops(B, H, N, D, True)
    peaks = measured_peaks()
    ach = tflops(f_nc, ms_nc)
    out = {
        "metric": f"attention bwd TFLOP/s at B={B},H={H},N={N},d={D} bf16", "value": tflops(f_nc + f_c, ms_nc + ms_c),
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": n_warm,
        "ms_per_step": ms_nc + ms_c, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"b{B}h{H}n{N}d{D} bf16 backward, non-causal + causal per step", "B": B, "H": H,
                   "N": N, "d": D, "scale": scale, "seed": SEED,
                   "flops": "10 B H N^2 d (five N x N x d products), halved for causal",
                   "l2": L2_NOTE, "statistic": "median over the timed steps"},
        "per_kernel": {"noncausal": {"ms_median": ms_nc, "ms_mean": statistics.fmean(t_nc),
                                     "tflops": tflops(f_nc, ms_nc)},
                       "causal": {"ms_median": ms_c, "ms_mean": statistics.fmean(t_c),
                                  "tflops": tflops(f_c, ms_c)}},
        "roofline": {"bound": "tensor", "kernel": "attn_bwd (prep + attn_bwd_kernel + dQ cast), non-causal",
                     "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": ach / peaks["bf16_tflops"], "traffic": None,
                     "algorithmic_flops_per_launch": f_nc},
        "gpu_launches": 6 * args.steps,
    }
    if sampler:
        out["clocks"] = summarize_clocks(sampler.samples, t0 - args.warmup_seconds, t1)
    print(json.dumps(out), flush=True)
    return 0


def run_fwd_shapes(args) -> int:
    """--fwd-shapes "B,H,N,d;...": the forward (non-causal, causal) on other problem
    sizes, one JSON line each, L2 flushed between launches. An extra measurement
    beside the headline line (the sequence sweep and the wide-head long problem)."""
    import torch

    from exact_attention_61_gb300 import attn, counts
    from gen import make_qkv

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    attn.load()
    peaks = measured_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(torch, dev, l2)
    stream = torch.cuda.current_stream(dev)
    for spec in args.fwd_shapes.split(";"):
        b_, h_, n_, d_ = (int(x) for x in spec.split(","))
        q, k, v = (t.to(dev) for t in make_qkv(b_, h_, n_, d_, DTYPE, SEED))
        o = torch.empty_like(q)
        lse = torch.empty((b_, h_, n_), dtype=torch.float32, device=dev)
        scale = 1.0 / math.sqrt(d_)
        res = {}
        for causal in (False, True):
            def launch():
                st = attn.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   b_, h_, n_, d_, causal, scale, attn.ATTN_BF16, stream.cuda_stream)
                if st != attn.ATTN_OK:
                    raise RuntimeError(f"attn_fwd failed: {attn.strerror(st)}")
            for i in range(max(args.warmup, 3)):
                flush(i)
                launch()
            ts = []
            for i in range(args.steps):
                flush(i)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch()
                e1.record(stream)
                ts.append((e0, e1))
            torch.cuda.synchronize(dev)
            ms = statistics.median(a.elapsed_time(b) for a, b in ts)
            f = counts.attn_flops(b_, h_, n_, d_, causal)
            res["causal" if causal else "noncausal"] = {"ms_median": ms, "tflops": tflops(f, ms),
                                                        "frac_of_peak": tflops(f, ms) / peaks["bf16_tflops"]}
        print(json.dumps({"metric": f"attention fwd TFLOP/s at B={b_},H={h_},N={n_},d={d_} bf16",
                          "unit": "TFLOP/s", "steps": args.steps, "dtype": "bf16", "data": "synthetic",
                          "l2": L2_NOTE, **res}), flush=True)
        del q, k, v, o, lse
    return 0


def _pct(xs, p):
    s = sorted(xs)
    return s[min(len(s) - 1, max(0, int(round(p / 100.0 * (len(s) - 1)))))]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--warmup-seconds", type=float, default=1.0,
                    help="keep warming up until the GPU has been busy this long")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work of the oracle baseline")
    ap.add_argument("--ref-step-seconds", type=float, default=2.0,
                    help="CPU work per step of the reference (oracle) arm")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-clocks", dest="clocks", action="store_false")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward pass instead (extra measurement, 1 GPU)")
    ap.add_argument("--bwd-shape", default="4,16,4096,64", metavar="B,H,N,d",
                    help="problem of --bwd (default: the headline problem)")
    ap.add_argument("--fwd-shapes", default=None, metavar="B,H,N,d;...",
                    help="time the forward on other sizes instead (extra measurement, 1 GPU)")
    ap.add_argument("--decode", default=None, metavar="NAME",
                    help="time a KV-cache decode workload instead (extra measurement, 1 GPU)")
    return ap.parse_args(argv)


def main(argv=None) -> int:
    args = parse_args(argv)
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")
    if args.impl == "reference":
        return run_reference(args)
    if args.decode:
        return run_decode(args)
    if args.bwd:
        return run_bwd(args)
    if args.fwd_shapes:
        return run_fwd_shapes(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
