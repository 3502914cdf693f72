#!/usr/bin/env python
"""Throughput of one MoE-layer forward on GB300 (and, on the side, of its backward).

A step is one pass of the whole path — route + per-chunk token counts,
index (counts, offsets, rows), permute, gate/up grouped GEMM with SwiGLU,
down grouped GEMM, gate-weighted combine — over one batch of T tokens, with inputs and packed
weights resident in HBM.  Default workload: one layer of the 951.9B model
(T=16,384 tokens, d=6,144, E=384 experts, top-8, f=1,792), seeded
synthetic inputs.  The working set (25 GB of weights, 201 MB of tokens)
is far larger than L2, so no flush is needed between steps.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]
With N > 1 every rank runs its own replica on its own GPU (weak scaling, no
collective on the data path; a barrier and a max over ranks around the
timed region); rank 0 prints one JSON line.  Under torchrun the ranks come
from the environment (WORLD_SIZE must equal N); otherwise bench.py starts N
local ranks itself.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MoE-layer fwd tokens/s and grouped-GEMM TFLOP/s (% bf16 peak); permute GB/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS_PER_STEP = 6  # route, index, permute, gate/up GEMM, down GEMM, combine
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")
GEMM_SOURCE = os.path.join(ROOT, "sparse_expert_gb300", "csrc", "grouped_gemm_2sm.cu")


# ----------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons every 50 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ------------------------------------------------------------------- peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


def code_sha256(path):
    """sha256 of a C++/CUDA source with its // comments and blank lines
    removed: counters recorded for a kernel stay valid across edits to its
    comments, and only those."""
    lines = []
    with open(path) as fh:
        for line in fh:
            code = line.split("//", 1)[0].rstrip()
            if code:
                lines.append(code)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the gate/up GEMM from a committed ncu summary,
    or None when absent or taken on a different kernel source."""
    try:
        with open(TRAFFIC_FILE) as fh:
            rec = json.load(fh)
    except (OSError, ValueError):
        return None
    if rec.get("workload") != workload or rec.get("source_code_sha256") != code_sha256(GEMM_SOURCE):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------- algorithmic work
def stage_work(cfg, counts=None, weight_bytes_per_value=2.0):
    """Algorithmic bytes / FLOPs per launch of each stage (real rows only).
    Given the token counts, the GEMMs also get their algorithmic bytes: the
    weights of every expert with rows (weight_bytes_per_value per weight:
    2 for bf16, codes plus scales for FP8) and their activations once."""
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    P = T * k
    work = {
        "route": {"bytes": T * E * 4 + P * 8},
        "index": {"bytes": P * 4 + P * 4 + 3 * P * 4 + E * 8},
        "permute": {"bytes": T * d * 2 + P * d * 2 + P * 4},
        "gate_up": {"flops": 4 * P * d * f},
        "down": {"flops": 2 * P * d * f},
        "combine": {"bytes": P * d * 2 + T * d * 2 + P * 4 + P * 4},   # rows, out, dest_row, gates
    }
    if counts is not None:
        nonempty = int((np.asarray(counts) > 0).sum())
        w = nonempty * d * f * weight_bytes_per_value
        work["gate_up"]["bytes"] = int(2 * w + P * d * 2 + P * f * 2)   # Wg, Wu; x_perm read, H written
        work["down"]["bytes"] = int(w + P * f * 2 + P * d * 2)          # Wd; H read, Y written
    return work


def backward_gemm_flops(cfg):
    """Algorithmic FLOPs of the GEMM stages of the layer backward (real rows
    only): the recomputed gate/up GEMM, two dgrad and two wgrad GEMMs (the
    down projection is not recomputed: the gate gradient comes from the dgrad
    down GEMM)."""
    P = cfg.T * cfg.k
    pdf = P * cfg.d * cfg.f
    return {"recompute_gate_up": 4 * pdf, "dgrad_down": 2 * pdf, "dgrad_gate_up": 4 * pdf, "wgrad_down": 2 * pdf,
            "wgrad_gate_up": 4 * pdf}


def weight_bytes_read(cfg, counts):
    nonempty = int((np.asarray(counts) > 0).sum())
    return nonempty * 3 * cfg.d * cfg.f * 2


# ------------------------------------------------------------ CPU oracle
def oracle_sample(cfg, x, logits, w_gate, w_up, w_down, tokens):
    """Host copies of what the oracle needs for a token sample: the sampled
    rows and the weights of every expert they route to."""
    import oracle
    idx, _ = oracle.route_topk(logits[tokens].cpu().numpy(), cfg.k, cfg.renormalize)
    experts = sorted(set(idx.reshape(-1).tolist()))

    class Host:
        def __init__(self, w):
            self.shape = tuple(w.shape)
            self.data = {e: w[e].float().cpu().numpy() for e in experts}

        def __getitem__(self, e):
            return self.data[int(e)]
    return (x[tokens].float().cpu().numpy(), logits[tokens].cpu().numpy(), Host(w_gate), Host(w_up), Host(w_down),
            len(experts))


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline_stages(cfg, x, logits, w_gate, w_up, w_down, n_tokens, n_experts):
    """The fp64 oracle on the host cores, stage by stage, on bounded samples
    of the workload (only the oracle calls are timed; fetching its inputs
    from the device is not):
      route, dispatch   every token;
      permute, combine  the first n_tokens tokens with their own dispatch
                        (the expert rows stand in for the expert outputs),
                        scaled by T / n_tokens;
      expert MLP        every row of n_experts experts spread over the
                        non-empty ones, scaled by P / rows sampled.
    Returns (seconds per stage, whether each is extrapolated, description)."""
    import oracle
    T, E, k = cfg.T, cfg.E, cfg.k
    P = T * k
    secs, extrap = {}, {}
    l_h = logits.cpu().numpy()
    t0 = time.perf_counter()
    idx, w = oracle.route_topk(l_h, k, cfg.renormalize)
    secs["route"], extrap["route"] = time.perf_counter() - t0, False
    t0 = time.perf_counter()
    counts, offsets, src, _ = oracle.dispatch(idx, E)
    secs["dispatch"], extrap["dispatch"] = time.perf_counter() - t0, False

    n = min(n_tokens, T)
    x_s = x[:n].double().cpu().numpy()
    _, _, src_s, dst_s = oracle.dispatch(idx[:n], E)
    t0 = time.perf_counter()
    xp = oracle.permute(x_s, src_s)
    t_perm = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.combine(xp, dst_s, w[:n])
    t_comb = time.perf_counter() - t0
    secs["permute"], secs["combine"] = t_perm * T / n, t_comb * T / n
    extrap["permute"] = extrap["combine"] = n < T
    del xp, x_s

    nonempty = np.nonzero(counts)[0]
    pick = nonempty[np.linspace(0, len(nonempty) - 1, min(n_experts, len(nonempty))).astype(np.int64)]
    mlp_s, rows = 0.0, 0
    for e in np.unique(pick):
        a, b = int(offsets[e]), int(offsets[e + 1])
        X = x[torch.from_numpy(src[a:b]).to(x.device)].double().cpu().numpy()
        wg = w_gate[e:e + 1].double().cpu().numpy()
        wu = w_up[e:e + 1].double().cpu().numpy()
        wd = w_down[e:e + 1].double().cpu().numpy()
        t0 = time.perf_counter()
        oracle.expert_mlp(X, np.array([0, b - a]), wg, wu, wd)
        mlp_s += time.perf_counter() - t0
        rows += b - a
        del X, wg, wu, wd
    secs["expert_mlp"], extrap["expert_mlp"] = mlp_s * P / max(rows, 1), rows < P
    desc = (f"fp64 numpy oracle stage by stage: route and dispatch of all {T} tokens; permute and combine of the "
            f"first {n} tokens x {T / n:.1f}; expert MLP of all {rows} rows of {len(np.unique(pick))} experts "
            f"x {P / max(rows, 1):.1f}")
    return secs, extrap, desc


SINGLE_THREAD_ORACLE = """
import sys, time
sys.path.insert(0, sys.argv[1])
import workloads, oracle
cfg = workloads.get("tiny")
inp = workloads.generate(cfg, 0)
args = (inp["x"].double().numpy(), inp["logits"].numpy(), inp["w_gate"].double().numpy(),
        inp["w_up"].double().numpy(), inp["w_down"].double().numpy(), cfg.k, cfg.renormalize)
oracle.moe_forward(*args)
t0 = time.perf_counter()
oracle.moe_forward(*args)
print(cfg.T / (time.perf_counter() - t0))
"""


def single_thread_tiny_oracle():
    """The whole oracle forward on the tiny workload in a child process whose
    BLAS and OpenMP pools hold one thread (tokens/s), or None if it fails."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[var] = "1"
    try:
        res = subprocess.run([sys.executable, "-c", SINGLE_THREAD_ORACLE, ROOT], env=env, capture_output=True,
                             text=True, timeout=300)
        return float(res.stdout.strip().splitlines()[-1]) if res.returncode == 0 else None
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        return None


def time_oracle(cfg, sample):
    import oracle
    x_rows, l_rows, wg, wu, wd, _ = sample
    t0 = time.perf_counter()
    oracle.moe_forward_tokens(x_rows, l_rows, wg, wu, wd, cfg.k, cfg.renormalize)
    return time.perf_counter() - t0


def stage_breakdown(moe, events, run_timed):
    """Per-stage mean times from as many steps as the timed region, run again
    after it, each with CUDA events at its stage boundaries (the timed region
    itself runs without them).  A short pass would not do: under the power cap
    the SM clock recovers in the idle gap before it, and a 20-step pass read
    gate/up 4 % faster than the steady state."""
    n = len(events)
    torch.cuda.synchronize()
    for s in range(n):
        run_timed(events[s])
    torch.cuda.synchronize()
    return {name: statistics.mean(events[s][i].elapsed_time(events[s][i + 1]) for s in range(n))
            for i, name in enumerate(moe.FORWARD_STAGES)}


def stage_table(stage_ms, work, peaks):
    """Per-stage ms with TFLOP/s and fraction of the bf16 peak (GEMMs) and/or
    GB/s and fraction of the HBM copy bandwidth (every stage with bytes)."""
    stages = {}
    for name, ms in stage_ms.items():
        st = {"ms": round(ms, 4)}
        if "flops" in work[name]:
            st["tflops"] = round(work[name]["flops"] / (ms * 1e-3) / 1e12, 2)
            st["frac_bf16_peak"] = round(st["tflops"] / peaks["bf16_tflops"], 4)
        if "bytes" in work[name]:
            st["gbs"] = round(work[name]["bytes"] / (ms * 1e-3) / 1e9, 1)
            st["frac_hbm"] = round(st["gbs"] / peaks["hbm_gbs"], 4)
        stages[name] = st
    return stages


def measure_workload(moe, name, seed, steps, warmup, world, local):
    """moe_forward of another seeded workload, timed like the headline (CUDA
    events on the launching stream, per-stage events, max over ranks)."""
    cfg = workloads.get(name)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    inp = workloads.generate(cfg, seed=seed, device="cuda")
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    x, logits = inp["x"], inp["logits"]
    del inp  # the unpacked weights
    ws = torch.empty(moe.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    nstage = len(moe.FORWARD_STAGES)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nstage + 1)] for _ in range(steps)]
    for _ in range(warmup):
        moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
    torch.cuda.synchronize()
    if moe.moe_read_device_status(ws) != 0:
        raise SystemExit(f"device status after the {name} warm-up")
    counts = moe.forward_intermediates(ws, T, E, k, d, f)["counts"].cpu().numpy()
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s_ in range(steps):
        moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if moe.moe_read_device_status(ws) != 0:
        raise SystemExit(f"device status after the {name} steps")
    max_s = max_over_ranks(t0.elapsed_time(t1) / 1e3, world, device="cuda")
    stage_ms = stage_breakdown(moe, events, lambda ev: moe.moe_forward_timed(
        x, logits, packed, E, k, f, ws, out, ev, cfg.renormalize, stream))
    peaks = load_peaks()
    work = stage_work(cfg, counts)
    stages = stage_table(stage_ms, work, peaks)
    gemm_ms = stage_ms["gate_up"] + stage_ms["down"]
    gemm_tf = (work["gate_up"]["flops"] + work["down"]["flops"]) / (gemm_ms * 1e-3) / 1e12
    return {
        "workload": f"{name}: T={T}, d={d}, E={E}, top-{k}, f={f}, {cfg.routing} routing, seed {seed}",
        "value": round(job_throughput(T * steps, world, max_s), 1), "unit": "tokens/s",
        "ms_per_step": round(max_s * 1e3 / steps, 4), "steps": steps, "warmup": warmup,
        "grouped_gemm": {"tflops": round(gemm_tf, 2), "frac_bf16_peak": round(gemm_tf / peaks["bf16_tflops"], 4),
                         "weight_bytes_read": weight_bytes_read(cfg, counts)},
        "permute_gbs": stages["permute"]["gbs"], "combine_gbs": stages["combine"]["gbs"],
        "experts_nonempty": int((counts > 0).sum()), "largest_group_rows": int(counts.max()),
        "stages": stages, "clocks": clk,
    }


# ------------------------------------------------------------------ arms
def gpu_arm(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    import sparse_expert_gb300 as moe

    cfg = workloads.get(args.workload)
    T, d, E, k, f = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f
    P = T * k
    inp = workloads.generate(cfg, seed=args.seed + rank, device="cuda")
    x, logits = inp["x"], inp["logits"]
    packed = moe.moe_pack_weights(inp["w_gate"], inp["w_up"], inp["w_down"])
    ws = torch.empty(moe.moe_forward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    nstage = len(moe.FORWARD_STAGES)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nstage + 1)] for _ in range(args.steps)]

    for _ in range(args.warmup):
        moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0, "device status after warm-up"
    inter = moe.forward_intermediates(ws, T, E, k, d, f)
    counts = inter["counts"].cpu().numpy()

    # events only at the GEMMs' boundaries (3: gate/up, 4: down, 5: combine): the roofline's kernel
    # time comes from the timed region itself, at the cost of three events a step; each is recorded
    # once here so that its handle exists before the timed region
    gemm_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for ev3 in gemm_ev:
        for e in ev3:
            e.record(stream)

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for s in range(args.steps):
        ev = [None] * (nstage + 1)
        ev[3], ev[4], ev[5] = gemm_ev[s]
        moe.moe_forward_timed(x, logits, packed, E, k, f, ws, out, ev, cfg.renormalize, stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    status = moe.moe_read_device_status(ws)
    if status != 0:
        raise SystemExit(f"device status {status} after the timed steps")
    max_s = max_over_ranks(elapsed_ms / 1e3, world, device="cuda")
    value = job_throughput(T * args.steps, world, max_s)

    region_ms = {"gate_up": statistics.mean(a.elapsed_time(b) for a, b, _ in gemm_ev),
                 "down": statistics.mean(b.elapsed_time(c) for _, b, c in gemm_ev)}
    stage_ms = stage_breakdown(moe, events, lambda ev: moe.moe_forward_timed(
        x, logits, packed, E, k, f, ws, out, ev, cfg.renormalize, stream))
    work = stage_work(cfg, counts)
    peaks = load_peaks()
    stages = stage_table(stage_ms, work, peaks)
    gemm_ms = stage_ms["gate_up"] + stage_ms["down"]
    gemm_tflops = (work["gate_up"]["flops"] + work["down"]["flops"]) / (gemm_ms * 1e-3) / 1e12
    dominant = max(("gate_up", "down"), key=lambda n: region_ms[n])
    achieved = work[dominant]["flops"] / (region_ms[dominant] * 1e-3) / 1e12
    traffic = recorded_traffic(args.workload) if dominant == "gate_up" else None
    roofline = {"bound": "tensor", "kernel": f"grouped_gemm_2sm_kernel ({dominant})", "achieved": round(achieved, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": traffic, "peak_source": f"bf16 dense burst, {peaks['source']}",
                "kernel_ms": round(region_ms[dominant], 4),
                "timing": "mean over the timed steps of the CUDA events recorded around the kernel inside them"}

    # the same layer with the permute fused into the gate/up GEMM (TMA gathers of x[src_token])
    gathered = None
    if not args.no_gathered:
        gev = [[torch.cuda.Event(enable_timing=True) for _ in range(nstage + 1)] for _ in range(args.steps)]
        for _ in range(args.warmup):
            moe.moe_forward_gathered(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
        torch.cuda.synchronize()
        barrier(world)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for s_ in range(args.steps):
            moe.moe_forward_gathered(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
        g1.record(stream)
        torch.cuda.synchronize()
        if moe.moe_read_device_status(ws) != 0:
            raise SystemExit("device status after the gathered forward")
        gat_s = max_over_ranks(g0.elapsed_time(g1) / 1e3, world, device="cuda")
        gstage = {name: round(ms, 4) for name, ms in stage_breakdown(moe, gev, lambda ev: moe.moe_forward_gathered_timed(
            x, logits, packed, E, k, f, ws, out, ev, cfg.renormalize, stream)).items() if name != "permute"}
        gathered = {"value": round(job_throughput(T * args.steps, world, gat_s), 1), "unit": "tokens/s",
                    "ms_per_step": round(gat_s * 1e3 / args.steps, 4), "stages_ms": gstage,
                    "gate_up_tflops": round(work["gate_up"]["flops"] / (gstage["gate_up"] * 1e-3) / 1e12, 1),
                    "note": "the same layer without x_perm: four warps of the gate/up GEMM gather its A rows "
                            "x[src_token[r]] with 16-byte cp.async copies; outputs bit-identical to the permuted "
                            "path"}

    # end to end: host buffers through the C ABI, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        # every step copies its batch in from pinned host memory and its output back, through
        # moe_forward_host_stream: copies on their own streams overlap the neighbouring steps' compute
        x_h = x.cpu().pin_memory()
        l_h = logits.cpu().pin_memory()
        o_h = torch.empty(T, d, dtype=torch.bfloat16).pin_memory()
        x_d = [torch.empty_like(x) for _ in range(2)]
        l_d = [torch.empty_like(logits) for _ in range(2)]
        o_d = [torch.empty_like(out) for _ in range(2)]
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        moe.moe_forward_host_stream([x_h] * max(3, args.warmup), [l_h] * max(3, args.warmup),
                                    [o_h] * max(3, args.warmup), x_d, l_d, o_d, packed, E, k, f, ws,
                                    cfg.renormalize, stream, cin, cout)
        barrier(world)
        t0 = time.perf_counter()
        moe.moe_forward_host_stream([x_h] * args.steps, [l_h] * args.steps, [o_h] * args.steps, x_d, l_d, o_d,
                                    packed, E, k, f, ws, cfg.renormalize, stream, cin, cout)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world, device="cuda")
        e2e = {"value": round(job_throughput(T * args.steps, world, e2e_s), 1), "unit": "tokens/s",
               "h2d_bytes_per_step": x_h.numel() * 2 + l_h.numel() * 4, "d2h_bytes_per_step": o_h.numel() * 2,
               "api": "moe_forward_host_stream (pinned host batches, copies overlapped with compute)"}

    # the same layer with FP8 (E4M3, blockwise fp32 scales) expert weights read by the GEMMs: each stage's codes
    # are dequantised in shared memory to exactly the bf16 values moe_dequantize_fp8_blockwise gives
    fp8 = None
    if not args.no_fp8:
        q = [moe.moe_quantize_fp8_blockwise(inp[n].reshape(-1)) for n in ("w_gate", "w_up", "w_down")]
        packed_fp8 = moe.moe_pack_weights_fp8(q[0], q[1], q[2], E, d, f)
        fp8_bytes = moe.moe_fp8_packed_weight_bytes(E, d, f)  # codes and scale records
        del q
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(nstage + 1)] for _ in range(args.steps)]
        for _ in range(args.warmup):
            moe.moe_forward_fp8(x, logits, packed_fp8, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
        torch.cuda.synchronize()
        fclocks = ClockSampler(local)
        fclocks.start()
        barrier(world)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for s_ in range(args.steps):
            moe.moe_forward_fp8(x, logits, packed_fp8, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=stream)
        f1.record(stream)
        torch.cuda.synchronize()
        fclk = fclocks.stop()
        if moe.moe_read_device_status(ws) != 0:
            raise SystemExit("device status after the FP8-weight forward")
        fp8_s = max_over_ranks(f0.elapsed_time(f1) / 1e3, world, device="cuda")
        fstage = stage_breakdown(moe, fev, lambda ev: moe.moe_forward_fp8_timed(
            x, logits, packed_fp8, E, k, f, ws, out, ev, cfg.renormalize, stream))
        fp8 = {"value": round(job_throughput(T * args.steps, world, fp8_s), 1), "unit": "tokens/s",
               "ms_per_step": round(fp8_s * 1e3 / args.steps, 4),
               "stages": stage_table(fstage, stage_work(cfg, counts, fp8_bytes / (3 * E * d * f)), peaks),
               "weight_bytes_read": fp8_bytes, "clocks": fclk,
               "note": "not the headline: weights stored as E4M3 codes with one fp32 scale per 128 values (lower "
                       "weight precision); the GEMMs dequantise each stage in shared memory, bit-identical to the "
                       "bf16 path on the dequantised weights, and read about half the weight bytes"}
        del packed_fp8

    # the same forward captured once into a CUDA graph and replayed: no host
    # work between steps and no launch gaps inside one
    graph_fwd = None
    if not args.no_graph:
        gstream = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(gstream):
            with torch.cuda.graph(graph, stream=gstream):
                moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out, stream=gstream)
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        if moe.moe_read_device_status(ws) != 0:
            raise SystemExit("device status after the graph replays")
        barrier(world)
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record()
        for _ in range(args.steps):
            graph.replay()
        g1.record()
        torch.cuda.synchronize()
        barrier(world)
        graph_s = max_over_ranks(g0.elapsed_time(g1) / 1e3, world, device="cuda")
        graph_fwd = {"value": round(job_throughput(T * args.steps, world, graph_s), 1), "unit": "tokens/s",
                     "ms_per_step": round(graph_s * 1e3 / args.steps, 4),
                     "note": "moe_forward captured once into a CUDA graph (torch.cuda.CUDAGraph) and replayed per step"}
        del graph

    # the routing stages alone on the same logits (route with softmax/top-k,
    # then the count/scan/index pass of moe_dispatch_scan: a histogram kernel
    # and the index kernel), each call captured `reps` times into a CUDA graph
    # and replayed, so no host work sits between the launches
    routing = None
    if not args.no_routing:
        reps = 50
        rws = torch.empty(moe.moe_dispatch_workspace_bytes(T, E, k), dtype=torch.uint8, device="cuda")
        ridx, rw = moe.moe_route_topk(logits, k, cfg.renormalize)
        torch.cuda.synchronize()

        def graph_us(call):
            gs = torch.cuda.Stream()
            with torch.cuda.stream(gs):
                for _ in range(3):
                    call(gs)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(gs):
                with torch.cuda.graph(g, stream=gs):
                    for _ in range(reps):
                        call(gs)
            # replays until the SM clock has settled at this workload's level (the
            # GEMM sections before leave it at the power-capped clock)
            for _ in range(200):
                g.replay()
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                best = min(best, a.elapsed_time(b) * 1e3 / reps)
            del g
            return best

        route_us = graph_us(lambda st: moe.moe_route_topk(logits, k, cfg.renormalize, stream=st))
        dispatch_us = graph_us(lambda st: moe.moe_dispatch_scan(ridx, E, topk_w=rw, workspace=rws, stream=st))

        # the same calls one at a time with L2 flushed before each (a 512 MB
        # buffer written, four times L2), CUDA events around the call alone;
        # the flush and a short spin keep the GPU busy while the host issues
        # the call, so the events time the kernels and not the host
        flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

        def flushed_us(call, n=20):
            times = []
            for _ in range(n + 2):
                flush.fill_(1)
                torch.cuda._sleep(100_000)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                call(stream)
                b.record(stream)
                torch.cuda.synchronize()
                times.append(a.elapsed_time(b) * 1e3)
            return statistics.median(times[2:])

        route_cold_us = flushed_us(lambda st: moe.moe_route_topk(logits, k, cfg.renormalize, stream=st))
        dispatch_cold_us = flushed_us(lambda st: moe.moe_dispatch_scan(ridx, E, topk_w=rw, workspace=rws, stream=st))
        del flush
        if moe.moe_read_device_status(rws) != 0:
            raise SystemExit("device status after the routing calls")
        rwork = stage_work(cfg)
        routing = {"route_us": round(route_us, 2), "dispatch_us": round(dispatch_us, 2),
                   "total_us": round(route_us + dispatch_us, 2),
                   "l2_flushed": {"route_us": round(route_cold_us, 2), "dispatch_us": round(dispatch_cold_us, 2),
                                  "total_us": round(route_cold_us + dispatch_cold_us, 2),
                                  "note": "one call at a time after writing a 512 MB buffer, median of 20"},
                   "route_gbs": round(rwork["route"]["bytes"] / (route_us * 1e-6) / 1e9, 1),
                   "route_frac_hbm": round(rwork["route"]["bytes"] / (route_us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                   "dispatch_gbs": round(rwork["index"]["bytes"] / (dispatch_us * 1e-6) / 1e9, 1),
                   "note": "moe_route_topk and moe_dispatch_scan (histogram + index kernels) alone on the workload's "
                           f"logits, best of 5 replays of a CUDA graph holding {reps} calls each, after 200 untimed "
                           "replays (the 26 MB of logits stay in L2 across the calls; l2_flushed has them cold); "
                           "the forward's route "
                           "stage also holds the workspace clear (a memset of its header and count table)"}
        del rws, ridx, rw

    # the dynamic tile schedule against a static one, with a kernel holding
    # 40 SMs on a second stream for the first half of every step (the
    # SonicMoE page's measurement, a dummy kernel occupying 40 SMs)
    contention = None
    if not args.no_contention:
        busy = 40
        side = torch.cuda.Stream()
        n_sms = torch.cuda.get_device_properties(local).multi_processor_count
        csteps = max(3, min(args.steps, 10))

        def timed(loaded, hold_ns):
            for _ in range(2):
                moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out)
            torch.cuda.synchronize()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(csteps + 1)]
            ev[0].record(stream)
            for i in range(csteps):
                if loaded:
                    # the occupier starts with the step: the side stream waits for the step boundary
                    side.wait_event(ev[i])
                    moe.moe_occupy_sms(busy, hold_ns, stream=side)
                moe.moe_forward(x, logits, packed, E, k, f, cfg.renormalize, workspace=ws, out=out)
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            return statistics.median(ev[i].elapsed_time(ev[i + 1]) for i in range(csteps))

        cres = {}
        hold_ns = 0
        for mode, name in ((moe.TILE_SCHEDULE_DYNAMIC, "dynamic"), (moe.TILE_SCHEDULE_STATIC, "static")):
            moe.moe_set_tile_schedule(mode)
            free_ms = timed(False, 0)
            if name == "dynamic":
                hold_ns = int(free_ms * 0.5e6)  # half of an unloaded step
            busy_ms = timed(True, hold_ns)
            cres[name] = {"ms_per_step": round(free_ms, 4), "ms_per_step_loaded": round(busy_ms, 4),
                          "slowdown": round(busy_ms / free_ms, 4)}
        moe.moe_set_tile_schedule(moe.TILE_SCHEDULE_DYNAMIC)
        if moe.moe_read_device_status(ws) != 0:
            raise SystemExit("device status after the contention steps")
        contention = {"busy_sms": busy, "sms": n_sms, "hold_ms": round(hold_ns / 1e6, 4),
                      # the step's SM-time lost to the occupier, as a fraction of the unloaded step
                      "sm_time_lost": round(busy * hold_ns / 1e6 / (n_sms * cres["dynamic"]["ms_per_step"]), 4),
                      **cres,
                      "note": "median step times; the occupier (moe_occupy_sms) holds busy_sms SMs for hold_ms from the "
                              "start of each step"}

    # the layer from the tokens: fused router (router GEMM + top-k) instead of given logits
    routed = None
    if not args.no_routed:
        wr = workloads.generate_router(cfg, seed=args.seed + rank, device="cuda")
        rp = moe.moe_pack_router_weights(wr)
        for _ in range(args.warmup):
            moe.moe_router_topk(x, rp, E, k, cfg.renormalize)
        # back to back between two events, like the steps: the host's per-call
        # work (outputs, tensor maps, launch) overlaps the previous kernel
        torch.cuda.synchronize()
        ra, rb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ra.record(stream)
        for _ in range(args.steps):
            moe.moe_router_topk(x, rp, E, k, cfg.renormalize)
        rb.record(stream)
        for _ in range(args.warmup):
            moe.moe_forward_routed(x, rp, packed, E, k, f, cfg.renormalize, workspace=ws, out=out)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            moe.moe_forward_routed(x, rp, packed, E, k, f, cfg.renormalize, workspace=ws, out=out)
        t1.record(stream)
        torch.cuda.synchronize()
        router_ms = ra.elapsed_time(rb) / args.steps
        routed_s = max_over_ranks(t0.elapsed_time(t1) / 1e3, world, device="cuda")
        router_tf = 2.0 * T * d * E / (router_ms * 1e-3) / 1e12
        routed = {"value": round(job_throughput(T * args.steps, world, routed_s), 1), "unit": "tokens/s",
                  "ms_per_step": round(routed_s * 1e3 / args.steps, 4),
                  "router_topk_ms": round(router_ms, 4), "router_tflops": round(router_tf, 1),
                  "note": "whole layer from x and router weights: fused router GEMM + top-k replaces the given logits"}

    # training use: the layer backward (forward recomputed inside it)
    backward = None
    if not args.no_backward:
        grads = {"dx": torch.empty(T, d, dtype=torch.bfloat16, device="cuda"),
                 "d_logits": torch.empty(T, E, dtype=torch.float32, device="cuda"),
                 "dw_gate": torch.empty(E, d, f, dtype=torch.bfloat16, device="cuda"),
                 "dw_up": torch.empty(E, d, f, dtype=torch.bfloat16, device="cuda"),
                 "dw_down": torch.empty(E, f, d, dtype=torch.bfloat16, device="cuda")}
        bws = torch.empty(moe.moe_backward_workspace_bytes(T, E, k, d, f), dtype=torch.uint8, device="cuda")
        dout = (torch.randn(T, d, device="cuda", generator=torch.Generator(device="cuda").manual_seed(args.seed + 5))
                * 0.1).to(torch.bfloat16)
        nb = len(moe.BACKWARD_STAGES)
        bsteps = max(1, min(args.steps, 20))
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(nb + 1)] for _ in range(bsteps)]
        for _ in range(max(3, min(args.warmup, 5))):
            moe.moe_backward_timed(x, logits, packed, dout, E, k, f, bws, grads, bev[0], cfg.renormalize, stream)
        torch.cuda.synchronize()
        bclocks = ClockSampler(local)
        bclocks.start()
        barrier(world)
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for s_ in range(bsteps):
            moe.moe_backward_timed(x, logits, packed, dout, E, k, f, bws, grads, bev[s_], cfg.renormalize, stream)
        b1.record(stream)
        torch.cuda.synchronize()
        bclk = bclocks.stop()
        if moe.moe_read_device_status(bws) != 0:
            raise SystemExit("device status after the backward steps")
        bwd_s = max_over_ranks(b0.elapsed_time(b1) / 1e3, world, device="cuda")
        bstage = {name: statistics.mean(bev[s_][i].elapsed_time(bev[s_][i + 1]) for s_ in range(bsteps))
                  for i, name in enumerate(moe.BACKWARD_STAGES)}
        bflops = backward_gemm_flops(cfg)
        bst = {}
        for name, ms in bstage.items():
            e = {"ms": round(ms, 4)}
            if name in bflops:
                e["tflops"] = round(bflops[name] / (ms * 1e-3) / 1e12, 1)
            bst[name] = e
        gemm_names = [n for n in moe.BACKWARD_STAGES if n in bflops]
        bgemm_ms = sum(bstage[n] for n in gemm_names)
        bdom = max(gemm_names, key=lambda n: bstage[n])
        bach = bflops[bdom] / (bstage[bdom] * 1e-3) / 1e12
        backward = {
            "value": round(job_throughput(T * bsteps, world, bwd_s), 1), "unit": "tokens/s",
            "ms_per_step": round(bwd_s * 1e3 / bsteps, 4), "steps": bsteps,
            "train_step_tokens_per_s": round(T / (max_s / args.steps + bwd_s / bsteps), 1),
            "gemm_tflops": round(sum(bflops.values()) / (bgemm_ms * 1e-3) / 1e12, 1),
            "stages": bst,
            "roofline": {"bound": "tensor", "kernel": f"grouped_gemm_bwd_kernel ({bdom})", "achieved": round(bach, 1),
                         "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                         "frac": round(bach / peaks["bf16_tflops_sustained"], 4), "traffic": None,
                         "peak_source": f"bf16 dense sustained, {peaks['source']}"},
            "clocks": bclk,
            "note": "gradients of x, the router logits and the three expert weight tensors for a given output "
                    "gradient; the forward is recomputed inside (route, index, permute, gate/up keeping G and U; the "
                    "gate gradient comes from the dgrad down GEMM, so the down projection is not recomputed); "
                    "train_step = forward + backward",
        }
        del bws, grads

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, extrap, desc = cpu_baseline_stages(cfg, x, logits, inp["w_gate"], inp["w_up"], inp["w_down"],
                                                 args.cpu_sample_tokens, args.cpu_sample_experts)
        total = sum(secs.values())
        cpu = {"value": round(T / total, 3), "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
               "sample": desc, "cpu_model": cpu_model(),
               "stages_s": {k_: round(v, 4) for k_, v in secs.items()},
               "extrapolated": sorted(k_ for k_, v in extrap.items() if v),
               "single_thread_tiny": {"value": single_thread_tiny_oracle(), "unit": "tokens/s", "cores": 1,
                                      "sample": "the whole oracle forward on the tiny workload (T=256, d=128, E=8, "
                                                "top-2, f=64), one BLAS/OpenMP thread"},
               "note": "value = T / the sum of the stage times (timed or scaled), one layer forward"}

    configs = None
    if not args.no_configs:
        # the other seeded workloads beside the headline one, each timed the same way
        del inp, x, logits, packed, ws, out, events
        torch.cuda.empty_cache()
        configs = {}
        for name in ("small", "skew", "long"):
            if name == args.workload:
                continue
            configs[name] = measure_workload(moe, name, args.seed + rank, max(3, min(args.steps, 20)),
                                             args.warmup, world, local)
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(max_s * 1e3 / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{args.workload}: MoE layer forward, T={T} tokens, d={d}, E={E} experts, "
                                   f"top-{k}, f={f}, bf16, fp32 router logits ({cfg.routing} routing), seed "
                                   f"{args.seed}",
                       "T": T, "d": d, "E": E, "k": k, "f": f, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (weights 3*E*d*f*2 bytes streamed every step)"},
            "grouped_gemm": {"tflops": round(gemm_tflops, 2), "frac_bf16_peak": round(gemm_tflops / peaks["bf16_tflops"], 4),
                             "weight_bytes_read": weight_bytes_read(cfg, counts)},
            "permute_gbs": stages["permute"]["gbs"],
            "stages": stages, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "routed_forward": routed,
            "gathered_forward": gathered, "fp8_weights_forward": fp8, "graph_forward": graph_fwd,
            "routing": routing, "contention": contention,
            "gpu_launches": KERNELS_PER_STEP * args.steps, "clocks": clk,
            "backward": backward, "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def reference_arm(args):
    """The fp64 oracle on the host cores, on samples of the same workload."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    cfg = workloads.get(args.workload)
    n = min(args.ref_sample_tokens, cfg.T)
    dev = f"cuda:{local}" if torch.cuda.is_available() else "cpu"
    inp = workloads.generate(cfg, seed=args.seed, device=dev)
    secs = []
    for s in range(args.warmup + args.steps):
        # step s: the oracle on n consecutive tokens; only the oracle call is timed
        tokens = (torch.arange(n) + (s * n) % max(1, cfg.T - n + 1)).to(dev)
        sample = oracle_sample(cfg, inp["x"], inp["logits"], inp["w_gate"], inp["w_up"], inp["w_down"], tokens)
        t = time_oracle(cfg, sample)
        if s >= args.warmup:
            secs.append(t)
        del sample
    total = sum(secs)
    value = n * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total * 1e3 / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: MoE layer forward, T={cfg.T} tokens, d={cfg.d}, E={cfg.E} "
                               f"experts, top-{cfg.k}, f={cfg.f}", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"each step: fp64 numpy oracle, full layer forward of {n} consecutive tokens"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _spawned_rank(rank, world, port, argv, arm):
    """Entry of a rank that bench.py started itself: the environment torchrun
    would have set, then the arm."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    arm(parse_args(argv))


def launch(args, argv, arm):
    """Runs `arm` on args.gpus ranks: the current process when it is already
    one rank of a torchrun job (WORLD_SIZE set) or when N = 1, else N local
    processes started here, one per GPU."""
    world_env = os.environ.get("WORLD_SIZE")
    if world_env is not None:
        if int(world_env) != args.gpus:
            raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world_env}: launch one rank per GPU")
        arm(args)
        return
    if args.gpus == 1:
        arm(args)
        return
    if arm is gpu_arm and torch.cuda.device_count() < args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but {torch.cuda.device_count()} CUDA devices are visible")
    import torch.multiprocessing as mp
    mp.spawn(_spawned_rank, args=(args.gpus, _free_port(), list(argv), arm), nprocs=args.gpus, join=True)


def parse_args(argv):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", choices=sorted(workloads.CONFIGS), default="t1")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-routed", action="store_true", help="skip the fused-router forward measurement")
    ap.add_argument("--no-backward", action="store_true", help="skip the layer-backward measurement")
    ap.add_argument("--no-gathered", action="store_true", help="skip the gathered (no x_perm) forward measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the other seeded workloads (small, skew, long)")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8-weight forward measurement")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay of the forward")
    ap.add_argument("--no-routing", action="store_true", help="skip the routing-only (route + dispatch) measurement")
    ap.add_argument("--no-contention", action="store_true",
                    help="skip the tile-schedule measurement beside a kernel holding 40 SMs")
    ap.add_argument("--cpu-sample-tokens", type=int, default=2048,
                    help="tokens of the CPU baseline's permute/combine sample")
    ap.add_argument("--cpu-sample-experts", type=int, default=16,
                    help="experts of the CPU baseline's expert-MLP sample")
    ap.add_argument("--ref-sample-tokens", type=int, default=4)
    args = ap.parse_args(argv)
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    return args


def main(argv=None, arm=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if arm is None:
        arm = reference_arm if args.impl == "reference" else gpu_arm
    launch(args, argv, arm)


if __name__ == "__main__":
    main()
