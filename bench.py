"""Benchmark of the dense projection GEMM step on GB300.

One step = forward, input gradient and weight gradient of the 4096 -> 12288
projection at T = 16384 tokens (BF16 operands, BF16 output, whole K per output
tile): Y = X W^T, dX = dY W, dW = dY^T X.  The metric is the step's BF16 TFLOP/s
(3 x 2*T*N*K FLOP) with per-op microseconds and the dominant kernel's fraction of
the measured dense BF16 peak.

Timing: W untimed warm-up steps, then K timed steps.  Before every step a buffer
of twice the L2 size is zeroed (cold L2, as in the pages' protocol); CUDA events
on the launching stream bracket each op, so the flush is not counted.  The timed
region is bracketed by a barrier and a device synchronize on both sides; the
reported time is the maximum over ranks.  With several GPUs each rank runs its
own replica of the workload ("scaling": "weak"); no data crosses ranks.

`--impl reference` times the FP64 CPU oracle (the slow plain definition) on the
host cores on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    python bench.py --suite cfg1,cfg2,cfg3,cfg4,cfg5     # per-op table of every configuration
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BF16 TFLOP/s & % tensor peak, 4096→12288 T=16384 fwd/dgrad/wgrad (µs)"
UNIT = "TFLOP/s"
T_TOK, N_OUT, K_IN = 16384, 12288, 4096
FLOP_OP = 2.0 * T_TOK * N_OUT * K_IN
WORKLOAD = "wide projection 4096->12288, T=16384, bf16 in/out, fwd+dgrad+wgrad"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(value: float) -> float:
    """The largest `value` over all ranks (the slowest rank sets a step's time)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(ms_per_step: float, world: int, flop_per_rank_step: float) -> float:
    """Whole-job throughput: every rank's FLOP over the slowest rank's step time."""
    return flop_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.window = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = rows
        if self.window:
            t0, t1 = self.window
            sel = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0]
            inside = sel or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "samples": len(inside), "reasons": reasons}


# ------------------------------------------------------------ GPU arm

def run_profile_case(args, local):
    """A small single-op case for ncu captures: one op, `--profile-T` tokens, a few GB.
    BF16 ops take N, K (default 4096 -> 12288); router ops FP32 operands (N default 256
    experts); batched ops `--profile-B` per-head problems of T x K -> N over [T, B, D]
    views."""
    import fp32_dense_projection_gb300 as dp
    from fp32_dense_projection_gb300 import build as dpbuild

    dpbuild.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dp.init(local)
    op, T = args.profile_op, args.profile_T
    router = op.startswith("router")
    batched = op.endswith("_batched")
    N = args.profile_N or (256 if router else N_OUT)
    K = args.profile_K or K_IN
    g = torch.Generator(device=device)
    g.manual_seed(7)
    out_dtype = torch.float32 if (args.profile_f32 or router) else torch.bfloat16
    if router:
        X = torch.randn(T, K, generator=g, device=device)
        W = torch.randn(N, K, generator=g, device=device) * 0.02
        dY = torch.randn(T, N, generator=g, device=device)
        a, b = {"router_fwd": (X, W), "router_dgrad": (dY, W), "router_wgrad": (dY, X)}[op]
        fn = {"router_fwd": dp.router_fwd, "router_dgrad": dp.router_dgrad, "router_wgrad": dp.router_wgrad}[op]
        call = lambda out=None: fn(a, b, out=out)
        plan = dp.plan(op, T, N, K, True)
    elif batched:
        B = args.profile_B
        X = torch.randn(T, B, K, generator=g, device=device).to(torch.bfloat16).permute(1, 0, 2)
        dY = torch.randn(T, B, N, generator=g, device=device).to(torch.bfloat16).permute(1, 0, 2)
        W = (torch.randn(B, N, K, generator=g, device=device) / 16.0).to(torch.bfloat16)
        base = op[:-len("_batched")]
        a, b = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (dY, X)}[base]
        fn = {"fwd": dp.dp_gemm_fwd_batched, "dgrad": dp.dp_gemm_dgrad_batched, "wgrad": dp.dp_gemm_wgrad_batched}[base]
        call = lambda out=None: fn(a, b, out=out, out_dtype=out_dtype)
        plan = dp.plan_batched(base, B, T, N, K, out_dtype == torch.float32)
    else:
        X = torch.randn(T, K, generator=g, device=device).to(torch.bfloat16)
        W = (torch.randn(N, K, generator=g, device=device) / 64.0).to(torch.bfloat16)
        dY = torch.randn(T, N, generator=g, device=device).to(torch.bfloat16)
        a, b = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (dY, X)}[op]
        fn = {"fwd": dp.dp_gemm_fwd, "dgrad": dp.dp_gemm_dgrad, "wgrad": dp.dp_gemm_wgrad}[op]
        call = lambda out=None: fn(a, b, out=out, out_dtype=out_dtype)
        plan = dp.plan(op, T, N, K, out_dtype == torch.float32)
    out = call()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    times = []
    for _ in range(args.steps):
        ev[0].record()
        call(out)
        ev[1].record()
        torch.cuda.synchronize()
        times.append(ev[0].elapsed_time(ev[1]))
    # each kernel's own duration as CUPTI records it: median of five calls, the 2xL2
    # buffer zeroed before each (the events above time whole calls, host enqueue included)
    from torch.profiler import ProfilerActivity, profile
    flush = torch.empty(2 * torch.cuda.get_device_properties(device).L2_cache_size, dtype=torch.uint8, device=device)
    with profile(activities=[ProfilerActivity.CUDA]):  # CUPTI warm-up: the first session can miss kernels
        flush.zero_()
        torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        for _ in range(5):
            flush.zero_()
            call(out)
        torch.cuda.synchronize()
    mine = ("gemm_bf16_kernel", "split_reduce_kernel", "split_x3_kernel", "router_ffma_kernel")
    kern = {}
    for e in prof.events():
        if e.device_type == torch.autograd.DeviceType.CUDA and any(k in e.name for k in mine):
            name = e.name.replace("(anonymous namespace)::", "").split("(")[0].replace("void ", "")
            kern.setdefault(name, []).append(e.time_range.end - e.time_range.start)
    assert dp.device_error() == 0
    flop = 2.0 * T * N * K * (args.profile_B if batched else 1)
    us = statistics.median(times) * 1e3
    return {"profile_case": op, "T": T, "N": N, "K": K, "B": args.profile_B if batched else 1,
            "out": "f32" if out_dtype == torch.float32 else "bf16",
            "us": round(us, 2), "tflops": round(flop / us / 1e6, 1),
            "kernel_us_cold_l2": {k: round(statistics.median(v), 1) for k, v in kern.items()}, "plan": plan}


def run_gpu(args, world, rank, local):
    import fp32_dense_projection_gb300 as dp
    from fp32_dense_projection_gb300 import build as dpbuild

    dpbuild.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    dp.init(local)

    # synthetic inputs generated on the device (seeded), same recipe shape as the tests
    g = torch.Generator(device=device)
    g.manual_seed(1234 + rank)
    X = torch.randn(T_TOK, K_IN, generator=g, device=device).to(torch.bfloat16)
    W = (torch.randn(N_OUT, K_IN, generator=g, device=device) / 64.0).to(torch.bfloat16)
    dY = torch.randn(T_TOK, N_OUT, generator=g, device=device).to(torch.bfloat16)
    Y = torch.empty(T_TOK, N_OUT, dtype=torch.bfloat16, device=device)
    dX = torch.empty(T_TOK, K_IN, dtype=torch.bfloat16, device=device)
    dW = torch.empty(N_OUT, K_IN, dtype=torch.bfloat16, device=device)
    ws = dp.Workspace(local)
    need = max(dp.workspace_size(op, T_TOK, N_OUT, K_IN) for op in ("fwd", "dgrad", "wgrad"))
    wsbuf = ws.get(need)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(max(2 * l2, 1 << 20), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    plans = {op: dp.plan(op, T_TOK, N_OUT, K_IN) for op in ("fwd", "dgrad", "wgrad")}
    launches_per_step = sum(kernel_launches(op, plans[op]) for op in plans)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        dp.dp_gemm_fwd(X, W, out=Y, workspace=wsbuf)
        if ev is not None:
            ev[1].record(stream)
        dp.dp_gemm_dgrad(dY, W, out=dX, workspace=wsbuf)
        if ev is not None:
            ev[2].record(stream)
        dp.dp_gemm_wgrad(dY, X, out=dW, workspace=wsbuf)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert dp.device_error() == 0, "kernel barrier timeout during warm-up"

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        step(events[i])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.time()
    sampler.mark(t0, t1)
    clocks = sampler.stop()
    per_op = {"fwd": [], "dgrad": [], "wgrad": []}
    for ev in events:
        per_op["fwd"].append(ev[0].elapsed_time(ev[1]))
        per_op["dgrad"].append(ev[1].elapsed_time(ev[2]))
        per_op["wgrad"].append(ev[2].elapsed_time(ev[3]))
    step_ms = [sum(per_op[k][i] for k in per_op) for i in range(args.steps)]
    ms_per_step = max_over_ranks(statistics.mean(step_ms))
    value = job_tflops(ms_per_step, world, 3 * FLOP_OP)

    # end to end through the public API with host buffers: pinned H2D of the
    # step's inputs, the three ops, D2H of the three results, all timed
    e2e = None
    e2e_steps = max(2, min(args.steps, 10))
    hX, hW, hdY = (t.cpu().pin_memory() for t in (X, W, dY))
    h2d = sum(t.numel() * t.element_size() for t in (hX, hW, hdY))
    d2h = sum(t.numel() * t.element_size() for t in (Y, dX, dW))

    # As a training loop prefetches its next batch: two sets of device buffers (and
    # of pinned host results) alternate between steps, so step k + 1's inputs go up
    # and step k's results come down while the other set's GEMMs run.  Within a step
    # X and W go up first, so the forward starts while dY (the largest input) is
    # still in flight, and each result comes back as soon as it exists.  Events
    # order everything: a set is refilled only after its previous step's GEMMs are
    # done with it, and its outputs are rewritten only after they have been read back.
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    sets = []
    for k in range(2):
        dev_set = (X, W, dY, Y, dX, dW) if k == 0 else tuple(torch.empty_like(t) for t in (X, W, dY, Y, dX, dW))
        host_out = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (Y, dX, dW))
        sets.append({"dev": dev_set, "host": host_out, "gemm_done": None, "down_done": None})

    def e2e_step(i):
        st = sets[i % 2]
        sX, sW, sdY, sY, sdX, sdW = st["dev"]
        hY, hdX, hdW = st["host"]
        ev = {k: torch.cuda.Event() for k in ("xw", "dy", "y", "dx", "dw", "gemm", "down")}
        with torch.cuda.stream(up):
            if st["gemm_done"] is not None:
                up.wait_event(st["gemm_done"])  # this set's previous GEMMs are done with its inputs
            sX.copy_(hX, non_blocking=True)
            sW.copy_(hW, non_blocking=True)
            ev["xw"].record(up)
            sdY.copy_(hdY, non_blocking=True)
            ev["dy"].record(up)
        if st["down_done"] is not None:
            stream.wait_event(st["down_done"])  # this set's previous results have been read back
        stream.wait_event(ev["xw"])
        dp.dp_gemm_fwd(sX, sW, out=sY, workspace=wsbuf)
        ev["y"].record(stream)
        stream.wait_event(ev["dy"])
        dp.dp_gemm_dgrad(sdY, sW, out=sdX, workspace=wsbuf)
        ev["dx"].record(stream)
        dp.dp_gemm_wgrad(sdY, sX, out=sdW, workspace=wsbuf)
        ev["dw"].record(stream)
        st["gemm_done"] = ev["dw"]
        with torch.cuda.stream(down):
            down.wait_event(ev["y"])
            hY.copy_(sY, non_blocking=True)
            down.wait_event(ev["dx"])
            hdX.copy_(sdX, non_blocking=True)
            down.wait_event(ev["dw"])
            hdW.copy_(sdW, non_blocking=True)
            ev["down"].record(down)
        st["down_done"] = ev["down"]

    for i in range(2):  # warm-up: both buffer sets
        e2e_step(i)
    torch.cuda.synchronize()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    ea.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(down)  # every download of every step is inside the timed region
    stream.wait_stream(up)
    eb.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(ea.elapsed_time(eb) / e2e_steps)
    e2e = {"value": round(job_tflops(e2e_ms, world, 3 * FLOP_OP), 2), "unit": UNIT,
           "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": e2e_steps}
    assert dp.device_error() == 0, "kernel barrier timeout during the timed region"

    peaks, peak_src = load_peaks()
    op_us = {k: statistics.median(v) * 1e3 for k, v in per_op.items()}
    dom = max(op_us, key=op_us.get)
    dom_mean_ms = statistics.mean(per_op[dom])
    achieved = FLOP_OP / (dom_mean_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    traffic = load_traffic(dom)
    roofline = {"bound": "tensor", "kernel": f"dp_gemm_{dom}", "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_src} (burst bf16)"}
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_TOK, "N": N_OUT, "K": K_IN, "out": "bf16",
                   "l2": "2xL2 buffer zeroed before every step (not timed); inputs also exceed L2",
                   "parallelism": f"replicas x{world}",
                   "plans": {k: {kk: plans[k][kk] for kk in ("block_n", "splits", "grid", "units")} for k in plans}},
        "per_op_us": {k: round(v, 2) for k, v in op_us.items()},
        "per_op_tflops": {k: round(FLOP_OP / (v * 1e-6) / 1e12, 1) for k, v in op_us.items()},
        "per_op_frac_of_peak": {k: round(FLOP_OP / (v * 1e-6) / 1e12 / peak, 4) for k, v in op_us.items()},
        "pages_context": {"dgrad_gb300_t16384_us": 811.6, "note": "pages' own GB300 figure, context only"},
        "roofline": roofline, "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(sample_rows=args.cpu_rows, single_rows=args.cpu_single_rows)
    if world > 1:
        torch.distributed.destroy_process_group()
    return result if rank == 0 else None


def kernel_launches(op: str, p: dict) -> int:
    """Kernels one call enqueues: the GEMM, the split reduction when the plan splits
    any tile, and the operand split of a router call."""
    split = p["splits"] > 1 and p["tiles_m"] * p["tiles_n"] > p["full_units"]
    return 1 + int(split) + int(str(op).startswith("router"))


def load_traffic(op: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    entry = d.get("kernels", {}).get(op)
    return entry.get("dram_bytes_per_launch") if entry else None


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp32_dense_projection_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".cpp", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------ CPU oracle

def oracle_sample(rows: int, seed: int = 0):
    """Time the FP64 oracle on `rows` output rows of each op of the workload."""
    import numpy as np

    import oracle
    from fp32_dense_projection_gb300 import inputs

    g = torch.Generator().manual_seed(seed)
    # only the operand rows the sampled outputs need are drawn in full
    X = inputs.normal((T_TOK, K_IN), seed, inputs.ROLE_X)
    W = inputs.normal((N_OUT, K_IN), seed, inputs.ROLE_W, 1.0 / 64)
    dY = inputs.normal((T_TOK, N_OUT), seed, inputs.ROLE_DY)
    oracle.build()
    rng = np.random.default_rng(seed)
    macs = 0
    t0 = time.perf_counter()
    r = rng.integers(0, T_TOK, rows)
    rr, cc = np.repeat(r, N_OUT), np.tile(np.arange(N_OUT), rows)
    oracle.fwd_bf16_at(X, W, rr, cc)
    macs += rr.size * K_IN
    rr, cc = np.repeat(r, K_IN), np.tile(np.arange(K_IN), rows)
    oracle.dgrad_bf16_at(dY, W, rr, cc)
    macs += rr.size * N_OUT
    rn = rng.integers(0, N_OUT, rows)
    rr, cc = np.repeat(rn, K_IN), np.tile(np.arange(K_IN), rows)
    oracle.wgrad_bf16_at(dY, X, rr, cc)
    macs += rr.size * T_TOK
    dt = time.perf_counter() - t0
    del g
    return 2.0 * macs / dt / 1e12, dt, oracle.num_threads()


def cpu_baseline(sample_rows: int, single_rows: int) -> dict:
    """The oracle on the host cores: all of them (OpenMP over output elements), and one
    thread in a child process (OMP_NUM_THREADS=1), each on its own bounded sample."""
    tflops, dt, cores = oracle_sample(sample_rows)
    out = {"value": round(tflops, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{sample_rows} output rows of each of fwd/dgrad/wgrad at the full 4096->12288 T=16384 "
                     f"shapes ({dt:.1f} s of FP64 CPU work on {cores} threads)"}
    if single_rows > 0:
        code = ("import json, bench; v, dt, c = bench.oracle_sample(%d, seed=5); "
                "print(json.dumps({'v': v, 'dt': dt, 'c': c}))" % single_rows)
        env = dict(os.environ, OMP_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
        if r.returncode == 0:
            d = json.loads(r.stdout.strip().splitlines()[-1])
            out["single_thread"] = {"value": round(d["v"], 6), "unit": UNIT, "cores": d["c"],
                                    "sample": f"{single_rows} output rows of each op ({d['dt']:.1f} s on one thread)"}
        else:
            out["single_thread"] = {"value": None, "error": (r.stderr or r.stdout).strip()[-300:]}
    return out


def run_reference(args, world, rank):
    if rank != 0:
        return None
    rows = max(1, args.cpu_rows // 8)
    for _ in range(args.warmup):
        oracle_sample(1, seed=1)
    vals, times = [], []
    for i in range(args.steps):
        v, dt, cores = oracle_sample(rows, seed=2 + i)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    sample = (f"{rows} output rows of each of fwd/dgrad/wgrad per step at the full shapes "
              f"({3 * rows} output rows, {statistics.median(times):.2f} s per step)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_TOK, "N": N_OUT, "K": K_IN,
                   "reference": "FP64 CPU oracle (plain definition), no GPU",
                   "step": f"a bounded sample of the workload: {sample}; value = the sample's FLOP / its time"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "kind": "oracle", "cores": cores,
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------------ measurement suite

def run_suite(args, local):
    """Every configuration of the workload set, per op, cold L2 before every call,
    timed three ways: CUDA events around an eager call, events around a CUDA-graph
    replay, and the kernel span of an eager call from the CUPTI trace (first start
    to last end of this library's kernels, excluding the launch latency that the
    events include).  Reported: microseconds, TFLOP/s, algorithmic GB/s and the
    fraction of the bounding roofline (tensor for arithmetic intensity above the
    ridge, HBM below).  One JSON line per case and timing."""
    import fp32_dense_projection_gb300 as dp
    from fp32_dense_projection_gb300 import build as dpbuild

    dpbuild.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dp.init(local)
    peaks, peak_src = load_peaks()
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ridge = tc_peak * 1e12 / (hbm_peak * 1e9)
    flush = torch.empty(2 * torch.cuda.get_device_properties(device).L2_cache_size, dtype=torch.uint8, device=device)
    ws = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(11)
    reps = args.suite_reps

    def eager(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)

    def graph(fn):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gr.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3)
        del gr
        return statistics.median(ts)

    def span(fn):
        # kernel span as a CUPTI trace records it: first start to last end of this
        # library's kernels in one call (cold L2 before each call), median over calls
        from torch.profiler import ProfilerActivity, profile
        fn()
        torch.cuda.synchronize()
        with profile(activities=[ProfilerActivity.CUDA]) as prof:
            for _ in range(reps):
                flush.zero_()
                fn()
            torch.cuda.synchronize()
        mine = ("gemm_bf16_kernel", "split_reduce_kernel", "split_x3_kernel", "router_ffma_kernel")
        calls, cur = [], None
        for e in sorted((e for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA),
                        key=lambda e: e.time_range.start):
            if any(k in e.name for k in mine):
                if cur is None:
                    cur = [e.time_range.start, e.time_range.end]
                else:
                    cur[1] = max(cur[1], e.time_range.end)
            elif cur is not None:
                calls.append(cur[1] - cur[0])
                cur = None
        if cur is not None:
            calls.append(cur[1] - cur[0])
        return statistics.median(calls) if calls else float("nan")

    def report(cfg, case, flop, tc_flop, nbytes, fn, plans=None):
        # flop: 2TNK of the op(s); tc_flop: tensor-pipe work (3x for BF16x3); nbytes: algorithmic bytes
        ai = tc_flop / nbytes
        bound = "tensor" if ai > ridge else "hbm"
        for mode, timer in (("eager", eager), ("graph", graph), ("kernel span", span)):
            us = timer(fn)
            us_repeat = timer(fn)  # the A/A repeat: the same measurement once more
            tflops = flop / us / 1e6
            gbs = nbytes / us / 1e3
            frac = (tc_flop / us / 1e6) / tc_peak if bound == "tensor" else gbs / hbm_peak
            line = {"suite": cfg, "case": case, "mode": mode, "us": round(us, 2), "us_repeat": round(us_repeat, 2),
                    "tflops": round(tflops, 1),
                    "gbs": round(gbs, 1), "bound": bound, "frac": round(frac, 3),
                    "of": f"{peak_src} {'bf16 burst' if bound == 'tensor' else 'HBM copy'} peak"}
            if plans:
                line["plan"] = plans
            print(json.dumps(line), flush=True)

    def plan_brief(op, T, N, K, f32):
        p = dp.plan(op, T, N, K, f32)
        return {k: p[k] for k in ("cta_pair", "block_n", "splits", "full_units", "swap_ab")}

    def bf(*shape, scale=1.0):
        return (torch.randn(*shape, generator=g, device=device) * scale).to(torch.bfloat16)

    def f32(*shape, scale=1.0):
        return torch.randn(*shape, generator=g, device=device) * scale

    def dense_ops(T, N, K, X, W, dY, od):
        e = 4 if od == torch.float32 else 2
        return {
            "fwd": (lambda: dp.dp_gemm_fwd(X, W, out_dtype=od, workspace=ws), 2 * T * K + 2 * N * K + e * T * N),
            "dgrad": (lambda: dp.dp_gemm_dgrad(dY, W, out_dtype=od, workspace=ws), 2 * T * N + 2 * N * K + e * T * K),
            "wgrad": (lambda: dp.dp_gemm_wgrad(dY, X, out_dtype=od, workspace=ws), 2 * T * N + 2 * T * K + e * N * K),
        }

    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]):  # CUPTI warm-up: the first session can miss kernels
        flush.zero_()
        torch.cuda.synchronize()
    which = set(args.suite.split(","))
    if "cfg1" in which:  # dense 4096 -> 1024 at T = 64, BF16 and FP32 output
        T, N, K = 64, 1024, 4096
        X, W, dY = bf(T, K), bf(N, K, scale=1 / 64), bf(T, N)
        for od, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
            for op, (fn, nb) in dense_ops(T, N, K, X, W, dY, od).items():
                report("cfg1", f"{op} T={T} {K}->{N} {name}", 2 * T * N * K, 2 * T * N * K, nb, fn,
                       plan_brief(op, T, N, K, od == torch.float32))
    if "cfg2" in which:  # FP32 router 4096 -> 256 at T in {64, 256, 1024}
        K, N = 4096, 256
        for T in (64, 256, 1024):
            X, W, dY = f32(T, K), f32(N, K, scale=0.02), f32(T, N)
            ops = {"router_fwd": (lambda: dp.router_fwd(X, W, workspace=ws), 4 * (T * K + N * K + T * N)),
                   "router_dgrad": (lambda: dp.router_dgrad(dY, W, workspace=ws), 4 * (T * N + N * K + T * K)),
                   "router_wgrad": (lambda: dp.router_wgrad(dY, X, workspace=ws), 4 * (T * N + T * K + N * K))}
            for op, (fn, nb) in ops.items():
                report("cfg2", f"{op} T={T}", 2 * T * N * K, 3 * 2 * T * N * K, nb, fn, plan_brief(op, T, N, K, True))
            del X, W, dY
    if "cfg3" in which:  # wide 4096 -> 12288, BF16 out
        N, K = 12288, 4096
        for T in (16384, 16231):
            X, W, dY = bf(T, K), bf(N, K, scale=1 / 64), bf(T, N)
            for op, (fn, nb) in dense_ops(T, N, K, X, W, dY, torch.bfloat16).items():
                report("cfg3", f"{op} T={T}", 2 * T * N * K, 2 * T * N * K, nb, fn, plan_brief(op, T, N, K, False))
            del X, W, dY
    if "cfg4" in which:  # thin-N weight gradient
        for T in (1025, 16173, 65537):
            Xf = bf(T, 5120)
            for K, N in ((4096, 64), (4096, 128), (4096, 512), (5120, 48), (5120, 64)):
                X = Xf[:, :K]
                dY = bf(T, N)
                for od, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
                    e = 4 if od == torch.float32 else 2
                    out = torch.empty(N, K, dtype=od, device=device)
                    fn = (lambda dY=dY, X=X, out=out, od=od: dp.dp_gemm_wgrad(dY, X, out=out, out_dtype=od, workspace=ws))
                    report("cfg4", f"wgrad T={T} {K}->{N} {name}", 2 * T * N * K, 2 * T * N * K,
                           2 * T * N + 2 * T * K + e * N * K, fn, plan_brief("wgrad", T, N, K, od == torch.float32))
            del Xf
    if "cfg5" in which:  # checkpointed step: fwd, recompute fwd, dgrad, wgrad
        for T in (1024, 4031, 16384):
            for N in (1024, 12288):
                K = 4096
                X, W, dY = bf(T, K), bf(N, K, scale=1 / 64), bf(T, N)
                Y = torch.empty(T, N, dtype=torch.bfloat16, device=device)
                dX = torch.empty(T, K, dtype=torch.bfloat16, device=device)
                dW = torch.empty(N, K, dtype=torch.bfloat16, device=device)

                def bwd(X=X, W=W, dY=dY, dX=dX, dW=dW):
                    # input and weight gradient: one co-scheduled launch or two calls, as planned
                    dp.dp_gemm_bwd(dY, X, W, dX=dX, dW=dW, workspace=ws)

                def bwd_two_calls(X=X, W=W, dY=dY, dX=dX, dW=dW):
                    dp.dp_gemm_dgrad(dY, W, out=dX, workspace=ws)
                    dp.dp_gemm_wgrad(dY, X, out=dW, workspace=ws)

                def step(X=X, W=W, dY=dY, Y=Y, dX=dX, dW=dW):
                    dp.dp_gemm_fwd(X, W, out=Y, workspace=ws)
                    dp.dp_gemm_fwd(X, W, out=Y, workspace=ws)
                    dp.dp_gemm_bwd(dY, X, W, dX=dX, dW=dW, workspace=ws)
                nb_b = (2 * T * N + 2 * N * K + 2 * T * K) * 2
                nb = 2 * (2 * T * K + 2 * N * K + 2 * T * N) + nb_b
                pb = dp.plan_bwd(T, N, K)
                form = {"co_scheduled": pb["fused"], "wgrad_first": pb["wgrad_first"],
                        "tile": [pb["dgrad"]["block_m"], pb["dgrad"]["block_n"]]}
                report("cfg5", f"bwd T={T} {K}->{N} bf16", 2 * 2 * T * N * K, 2 * 2 * T * N * K, nb_b, bwd, form)
                report("cfg5", f"bwd T={T} {K}->{N} bf16 two calls", 2 * 2 * T * N * K, 2 * 2 * T * N * K, nb_b,
                       bwd_two_calls)
                report("cfg5", f"2fwd+bwd T={T} {K}->{N} bf16", 4 * 2 * T * N * K, 4 * 2 * T * N * K, nb, step, form)
                del X, W, dY, Y, dX, dW
            K, N = 4096, 256
            X, W, dY = f32(T, K), f32(N, K, scale=0.02), f32(T, N)
            Y, dX, dW = torch.empty(T, N, device=device), torch.empty(T, K, device=device), torch.empty(N, K, device=device)

            def rbwd(X=X, W=W, dY=dY, dX=dX, dW=dW):
                dp.router_dgrad(dY, W, out=dX, workspace=ws)
                dp.router_wgrad(dY, X, out=dW, workspace=ws)

            def rstep(X=X, W=W, dY=dY, Y=Y, dX=dX, dW=dW):
                dp.router_fwd(X, W, out=Y, workspace=ws)
                dp.router_fwd(X, W, out=Y, workspace=ws)
                dp.router_dgrad(dY, W, out=dX, workspace=ws)
                dp.router_wgrad(dY, X, out=dW, workspace=ws)
            nb = 4 * (2 * (T * K + N * K + T * N) + 2 * (T * N + N * K + T * K))
            report("cfg5", f"router bwd T={T} {K}->{N} f32", 2 * 2 * T * N * K, 3 * 2 * 2 * T * N * K,
                   4 * 2 * (T * N + N * K + T * K), rbwd)
            report("cfg5", f"router 2fwd+bwd T={T} {K}->{N} f32", 4 * 2 * T * N * K, 3 * 4 * 2 * T * N * K, nb, rstep)
            del X, W, dY, Y, dX, dW
    if "batched" in which:  # per-head projections, 128 heads, T = 4096: one batched launch vs 128 calls
        H, T = 128, 4096
        for N, K in ((512, 128), (128, 512)):
            for op in ("fwd", "dgrad", "wgrad"):
                X = bf(T, H, K).permute(1, 0, 2)              # [H, T, K] per-head views of [T, H, K]
                dY = bf(T, H, N).permute(1, 0, 2)
                W = bf(H, N, K, scale=1 / 16)
                fb = {"fwd": lambda: dp.dp_gemm_fwd_batched(X, W, workspace=ws),
                      "dgrad": lambda: dp.dp_gemm_dgrad_batched(dY, W, workspace=ws),
                      "wgrad": lambda: dp.dp_gemm_wgrad_batched(dY, X, workspace=ws)}[op]
                single = {"fwd": lambda: [dp.dp_gemm_fwd(X[h], W[h], workspace=ws) for h in range(H)],
                          "dgrad": lambda: [dp.dp_gemm_dgrad(dY[h], W[h], workspace=ws) for h in range(H)],
                          "wgrad": lambda: [dp.dp_gemm_wgrad(dY[h], X[h], workspace=ws) for h in range(H)]}[op]
                nb = H * (2 * T * K + 2 * N * K + 2 * T * N)
                report("batched", f"{op} {H} heads T={T} {K}->{N} batched", H * 2 * T * N * K, H * 2 * T * N * K,
                       nb, fb, plan_brief_b(op, H, T, N, K))
                report("batched", f"{op} {H} heads T={T} {K}->{N} {H} single calls", H * 2 * T * N * K,
                       H * 2 * T * N * K, nb, single)
                del X, dY, W
    assert dp.device_error() == 0


def plan_brief_b(op, B, T, N, K):
    import fp32_dense_projection_gb300 as dp
    p = dp.plan_batched(op, B, T, N, K)
    return {k: p[k] for k in ("cta_pair", "block_n", "splits", "full_units", "swap_ab", "tiles")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=160, help="oracle sample on all host cores (~10 s on 16)")
    ap.add_argument("--cpu-single-rows", type=int, default=10, help="oracle sample on one thread (~7 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-op", default=None,
                    choices=["fwd", "dgrad", "wgrad", "router_fwd", "router_dgrad", "router_wgrad",
                             "fwd_batched", "dgrad_batched", "wgrad_batched"],
                    help="run only a single-op case (for ncu captures); prints each kernel's CUPTI duration "
                         "after a cold L2 as kernel_us_cold_l2")
    ap.add_argument("--profile-T", type=int, default=4096)
    ap.add_argument("--profile-N", type=int, default=0)
    ap.add_argument("--profile-K", type=int, default=0)
    ap.add_argument("--profile-f32", action="store_true")
    ap.add_argument("--profile-B", type=int, default=128, help="batched profile cases: problems (heads)")
    ap.add_argument("--suite", default=None,
                    help="comma list of cfg1..cfg5 (and 'batched'): per-op eager/graph/kernel-span measurements")
    ap.add_argument("--suite-reps", type=int, default=10)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_env()
    if args.suite:
        run_suite(args, local)
        return
    if args.profile_op:
        print(json.dumps(run_profile_case(args, local)), flush=True)
        return
    if args.impl == "reference":
        out = run_reference(args, world, rank)
    else:
        out = run_gpu(args, world, rank, local)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
