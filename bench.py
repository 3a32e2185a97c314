"""Benchmark of the streaming Sinkhorn hot path on one GB300 (or N replicas).

One step = the whole hot path over one synthetic problem: preparation,
every Sinkhorn iteration of the workload's eps schedule (from a cold start),
then its plan operator (barycentric projection, grad_x or P V).  Prints one
JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the float64 CPU oracle, bounded sample

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the stream the library launches on; a 256 MB buffer is written between
steps to flush the 129 MB L2.  The half-update kernel is also timed launch by
launch with the library's own events (fs_timing_*) over the same region; that
gives the roofline numbers.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from streaming_sinkhorn_solver_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

METRIC = "Sinkhorn iters/s and score-pairs/s at n=m=50k (d=3/64/512); % of roofline"
DEFAULT_WORKLOAD = "c4_n50k_d512"
PROFILES = os.path.join(ROOT, "profiles")
# ex2 rate of the special-function units on sm_103 (per SM per clock, measured)
# and the FP32 lanes per SM per clock; the ALU roofline is the slower of the
# two limits, times the SM count and the SM clock.
EX2_PER_CLK_SM = 32
FP32_LANES_PER_CLK_SM = 128


def fp32_ops_per_pair(d: int, tensor_path: bool) -> int:
    """FP32 lane-ops one score pair needs at the least: on the FMA path d
    fused multiply-adds (the column bias, with the row's exponent offset
    folded into it, is the chain's first addend) and one accumulation; on the
    tensor path the dot product and the offset are on the tensor pipe and the
    epilogue keeps the scale-and-bias multiply-add and the sum."""
    return 2 if tensor_path else d + 1


def tensor_peak(peaks: dict, sm_mhz: float):
    """Dense f16/bf16 tensor peak for a kernel that ran at median SM clock
    `sm_mhz`: the measured sustained cuBLAS rate, scaled from the median SM
    clock it was measured at to the run's clock (the tensor pipe's work per
    clock is fixed, so a run at a higher clock than the power-capped
    measurement has a proportionally higher ceiling).  Without a recorded
    clock the burst rate is used.  Returns (TFLOP/s, description)."""
    sustained = float(peaks["bf16_tflops_sustained"])
    at = ((peaks.get("clocks_under_load") or {}).get("sm_mhz_median"))
    if at and sm_mhz:
        peak = sustained * float(sm_mhz) / float(at)
        return peak, (f"{peaks['source']} bf16 dense sustained {sustained:.1f} TFLOP/s at a median "
                      f"{float(at):.0f} MHz, scaled to the run's median {float(sm_mhz):.0f} MHz; "
                      f"f16 operands have the same nominal rate")
    burst = float(peaks["bf16_tflops"])
    return burst, (f"{peaks['source']} bf16 dense burst (no clock recorded for the sustained "
                   f"figure); f16 operands have the same nominal rate")


def _rank_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, tag: str = ""):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples go to FS_CLOCK_LOG_DIR when set (to keep them), else
        # to the temporary directory; the JSON line carries their summary
        log_dir = os.environ.get("FS_CLOCK_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_gpu{gpu_index}{tag}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# Sources that define and launch the dominant half-update kernel of each path
# (kernel, host launch code and the headers they share): a committed ncu
# summary stays valid while none of these files changes.
KERNEL_SOURCES = {
    "fma": ["fs_fma.cu", "fs_fma_host.cu", "fs_api.cu", "fs_internal.cuh", "fs_host.cuh",
            "fs_shard.cuh"],
    "tc": ["fs_tc_ref.cu", "fs_tc_half.cu", "fs_tc_host.cu", "fs_tc.cuh", "fs_tc_kernels.cuh",
           "fs_internal.cuh", "fs_host.cuh", "fs_shard.cuh"],
    "pair": ["fs_tc_pair.cu", "fs_tc_host.cu", "fs_tc.cuh", "fs_tc_kernels.cuh", "fs_internal.cuh",
             "fs_host.cuh", "fs_shard.cuh"],
    "sparse": ["fs_sparse.cu", "fs_internal.cuh", "fs_host.cuh"],
}


def kernel_family(d: int, tensor_path: bool) -> str:
    if not tensor_path:
        return "fma"
    return "tc" if d <= 128 else "pair"


def _code_only(text: str) -> str:
    """C++ source without its comments and blank lines, each line stripped:
    a change to a comment alone leaves the hash below unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


def _kernel_source_hash(family: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "streaming_sinkhorn_solver_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[family]):
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            h.update(name.encode())
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic_from_profiles(workload: str, family: str):
    """DRAM bytes per launch of the half-update kernel from the committed ncu
    summary for this workload, or None if absent or taken on other sources."""
    path = os.path.join(PROFILES, f"half_update_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if line.startswith("- ") and "=" in line:
            k, v = line[2:].split("=", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_hash") != _kernel_source_hash(family):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def replica_seed(w, rank: int) -> int:
    """Weak scaling: rank r solves its own replica, drawn with seed + r."""
    return WORKLOADS[w.name].seed + rank


def max_over_ranks(x: float, device=None) -> float:
    """The largest value over the ranks of the default process group (the job
    is as slow as its slowest rank); x itself outside a group of > 1 ranks."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(world: int, units_per_rank_step: float, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank_step * steps / (total_ms * 1e-3)


def _work(w, n, m, d):
    """Algorithmic work of one step."""
    iters = w.n_iter
    pairs = 2 * n * m * iters + (n * m if w.apply else 0)
    return iters, pairs


def _step_fn(fs, w, t, path):
    import torch

    def step(host=None):
        src = host if host is not None else t
        g0 = src["g0"]
        if host is None:
            g0.zero_()
        f, g = src["f"], g0
        for eps, iters in w.stages:
            fs.fs_sinkhorn_solve(src["X"], src["a"], src["Y"], src["b"], eps, iters, f, g, path=path)
        eps_last = w.stages[-1][0]
        if w.apply == "barycentric":
            fs.fs_barycentric(src["X"], src["a"], src["Y"], src["b"], eps_last, f, g, src["out"],
                              path=path)
        elif w.apply == "grad_x":
            fs.fs_grad_x(src["X"], src["a"], src["Y"], src["b"], eps_last, f, g, src["out"], path=path)
        elif w.apply == "pv":
            fs.fs_apply_plan(src["X"], src["a"], src["Y"], src["b"], eps_last, f, g, src["V"],
                             src["out"], path=path)
        return f, g
    return step


def _cpu_baseline(w, inp, seconds: float):
    """The float64 oracle as it stands, on a bounded sample of this workload:
    f-updates of a stated number of rows against all m columns."""
    import oracle as orc
    n, m, d = w.n, w.m, w.d
    eps = w.stages[0][0]
    g = np.zeros(m)
    # size the sample from a short probe so the timed part takes ~`seconds`
    probe_rows = np.arange(min(n, max(4, orc.num_threads())), dtype=np.int64)
    t0 = time.perf_counter()
    orc.f_update_rows(inp["X"], inp["Y"], inp["b"], eps, g, probe_rows)
    dt = max(time.perf_counter() - t0, 1e-6)
    rows_n = int(min(n, max(len(probe_rows), len(probe_rows) * seconds / dt)))
    rows = np.linspace(0, n - 1, rows_n).astype(np.int64)
    reps = 0
    t0 = time.perf_counter()
    while True:  # repeat the sample (a row set is at most all n rows) until `seconds`
        orc.f_update_rows(inp["X"], inp["Y"], inp["b"], eps, g, rows)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 0.8 * seconds or rows_n < n:
            break
    pairs = reps * rows_n * m
    return {"value": pairs / dt, "unit": "score-pairs/s", "cores": orc.num_threads(),
            "kind": "oracle",
            "sample": f"{reps} x float64 f-update of {rows_n} evenly spaced rows against all {m} "
                      f"columns (d={d}), {dt:.1f} s; the full step is {_work(w, n, m, d)[1]:.3e} pairs"}


def arm_config(w) -> dict:
    """The workload's `config` object, the same for both arms."""
    n, m, d = w.n, w.m, w.d
    big = (n + m) * d * 4 > 129e6
    if w.tau > 0:
        eps, iters = w.stages[0]
        return {"workload": w.name, "n": n, "m": m, "d": d, "eps": eps, "iters": iters,
                "coarse_iters": w.coarse_iters, "tau": w.tau,
                "l2": "256 MB write between timed steps; inputs also > L2"}
    return {"workload": w.name, "n": n, "m": m, "d": d,
            "stages": [list(st) for st in w.stages], "apply": w.apply,
            "l2": "256 MB write between timed steps; inputs also > L2" if big
                  else "256 MB write between timed steps"}


def run_reference(args, w):
    """The reference arm: the oracle, timed on the host cores."""
    rank, world, _ = _rank_info()
    if rank != 0:
        return
    import oracle as orc
    inp = make_inputs(w.name)
    n, m, d = w.n, w.m, w.d
    eps = w.stages[0][0]
    g = np.zeros(m)
    rows_per_step = max(orc.num_threads(), int(args.ref_rows))
    times = []
    rows_all = np.random.default_rng(0).permutation(n)
    for s in range(args.warmup + args.steps):
        rows = np.sort(rows_all[(s * rows_per_step) % n:][:rows_per_step]).astype(np.int64)
        t0 = time.perf_counter()
        orc.f_update_rows(inp["X"], inp["Y"], inp["b"], eps, g, rows)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    tot = sum(times)
    pairs = rows_per_step * m * args.steps
    value = pairs / tot
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "score-pairs/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": arm_config(w),
            "cpu_baseline": {"value": value, "unit": "score-pairs/s", "cores": orc.num_threads(),
                             "kind": "oracle",
                             "sample": f"per step: float64 f-update of {rows_per_step} rows "
                                       f"against all {m} columns"},
            "e2e": {"value": value, "unit": "score-pairs/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _dense_roofline(w, path, half_ms, half_n, rates, clocks, sms):
    """Roofline of the dense half-update from its own events.  Per launch (one
    f- or g-update) the algorithmic work is n*m score pairs: 2 n m d tensor
    flops (tensor path), n m exponentials with d + 1 (FMA path) or 2 (tensor
    path) FP32 lane-ops each, and the streamed operand bytes; the binding term
    is the largest of the three times."""
    n, m, d = w.n, w.m, w.d
    peaks = _peaks()
    tensor_path = (path == "tensor") or (path == "auto" and d > 16)
    avg_half_ms = half_ms / max(half_n, 1)
    t_launch = avg_half_ms * 1e-3
    pairs_per_half = n * m
    clk = (clocks or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    ex2_clk = rates.get("ex2_per_clk_sm") or EX2_PER_CLK_SM
    fp32_clk = rates.get("fma2_lanes_per_clk_sm") or FP32_LANES_PER_CLK_SM
    rate_src = "measured by fs_unit_rates" if "ex2_per_clk_sm" in rates else "nominal"
    ex2_peak = ex2_clk * sms * clk * 1e6                               # ex2 / s
    fp32_ops = fp32_ops_per_pair(d, tensor_path)
    fp32_pair_peak = fp32_clk / fp32_ops * sms * clk * 1e6             # pairs / s
    tflops_peak, tflops_src = tensor_peak(peaks, clk)
    hbm_peak = float(peaks["hbm_gbs"])
    op_bytes = 2 if tensor_path else 4
    alg_bytes = op_bytes * (n + m) * d + 4 * 3 * (n + m)                # operands + biases/outputs
    alu_peak = min(ex2_peak, fp32_pair_peak)                           # pairs / s
    terms = {"alu_s": pairs_per_half / alu_peak, "hbm_s": alg_bytes / (hbm_peak * 1e9)}
    if tensor_path:
        terms["tensor_s"] = 2.0 * pairs_per_half * d / (tflops_peak * 1e12)
    bound = max(terms, key=terms.get)[:-2]
    if bound == "tensor":
        achieved = 2.0 * pairs_per_half * d / t_launch / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tflops_peak, "unit": "TFLOP/s",
                "peak_source": tflops_src,
                "frac_of_burst": achieved / float(peaks["bf16_tflops"])}
    elif bound == "alu":
        achieved = pairs_per_half / t_launch / 1e9
        per_clk = min(ex2_clk, fp32_clk / fp32_ops)
        roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak / 1e9, "unit": "Gpair/s",
                "peak_source": f"derived: min(MUFU {ex2_clk:.1f} ex2/clk/SM, FP32 "
                               f"{fp32_clk:.1f} lanes/clk/SM / {fp32_ops} lane-ops per "
                               f"pair) = {per_clk:.1f} pairs/clk/SM ({rate_src}) x {sms} SMs x "
                               f"{clk:.0f} MHz (median SM clock sampled in the timed region)",
                "mufu_frac": achieved * 1e9 / ex2_peak,
                "fp32_frac": achieved * 1e9 / fp32_pair_peak}
    else:
        achieved = alg_bytes / t_launch / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "peak_source": f"{peaks['source']} copy bandwidth"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = _traffic_from_profiles(w.name, kernel_family(d, tensor_path))
    roof["kernel"] = "half_update"
    roof["avg_launch_ms"] = avg_half_ms
    roof["launches"] = half_n
    roof["roofline_ms"] = {k[:-2]: v * 1e3 for k, v in terms.items()}
    roof["algorithmic_bytes_per_launch"] = alg_bytes
    roof["unit_rates"] = dict(rates, source=rate_src)
    return roof


# The metric's other points (n = m = 50k at d = 3 and d = 64) and the other
# configurations of the workload set (c5 at d = 1024, c2 at 10k, c1), each
# measured after the timed region of the default workload (d = 512) in the
# same process.
METRIC_POINTS = ("c2_n50k_d3", "c3_n50k_d64", "c5_n20k_m30k_d1024", "c2_n10k_d3", "c1_n512_d2")
# every point is timed over at least this many steps and about this long, so
# that its clock record holds several samples (nvidia-smi samples every 200 ms)
POINT_MIN_STEPS = 10
POINT_MIN_MS = 2500.0
POINT_MAX_STEPS = 5000


def point_steps(warm_ms_per_step: float) -> int:
    """Timed steps of a metric point from its warm-up step time."""
    want = int(POINT_MIN_MS / max(warm_ms_per_step, 1e-3)) + 1
    return max(POINT_MIN_STEPS, min(POINT_MAX_STEPS, want))


def _metric_point(fs, name, dev, rates, path, warmup=3):
    """One more workload, timed like the main one (warm-up, CUDA events
    around each step on the launching stream, a 256 MB write between steps,
    the half-update's own events for the roofline), over point_steps()
    steps."""
    import torch
    w = WORKLOADS[name]
    n, m, d = w.n, w.m, w.d
    inp = make_inputs(w.name)
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    t["f"] = torch.empty(n, device=dev)
    t["g0"] = torch.zeros(m, device=dev)
    t["out"] = torch.empty(n, w.k if w.apply == "pv" else d, device=dev) if w.apply else None
    step = _step_fn(fs, w, t, path)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(warmup):
        if i == warmup - 1:
            w0.record(stream)
        step()
    w1.record(stream)
    torch.cuda.synchronize()
    steps = point_steps(w0.elapsed_time(w1))
    sampler = ClockSampler(dev.index, tag=f"_{name}")
    sampler.start()
    fs.fs_timing_read()
    fs.fs_timing_enable(True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s_ in range(steps):
        flush.fill_(float(s_))
        ev[s_][0].record(stream)
        step()
        ev[s_][1].record(stream)
    torch.cuda.synchronize()
    fs.fs_timing_enable(False)
    (half_ms, _, _), (half_n, _, _) = fs.fs_timing_read()
    clocks = sampler.stop()
    total_ms = sum(a.elapsed_time(b) for a, b in ev)
    iters, pairs = _work(w, n, m, d)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    roof = _dense_roofline(w, path, half_ms, half_n, rates, clocks, sms)
    keep = ("bound", "achieved", "peak", "unit", "frac", "mufu_frac", "fp32_frac", "frac_of_burst",
            "traffic", "avg_launch_ms", "launches")
    return {"workload": name, "n": n, "m": m, "d": d, "steps": steps, "warmup": warmup,
            "value": pairs * steps / (total_ms * 1e-3), "unit": "score-pairs/s",
            "iters_per_s": iters * steps / (total_ms * 1e-3), "ms_per_step": total_ms / steps,
            "roofline": {k: roof[k] for k in keep if k in roof}, "clocks": clocks}


def run_gb300(args, w):
    import torch
    from streaming_sinkhorn_solver_gb300 import binding as fs

    rank, world, local = _rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    fs.load_library()
    n, m, d = w.n, w.m, w.d
    # weak scaling: every rank solves its own replica of the workload
    inp = make_inputs(w.name, seed=replica_seed(w, rank))
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    k_out = w.k if w.apply == "pv" else d
    t["f"] = torch.empty(n, device=dev)
    t["g0"] = torch.zeros(m, device=dev)
    t["out"] = torch.empty(n, k_out, device=dev) if w.apply else None
    path = args.path
    step = _step_fn(fs, w, t, path)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB > L2

    stream = torch.cuda.current_stream()
    try:
        rates = fs.fs_unit_rates()
    except Exception as exc:  # pragma: no cover - reported, nominal rates used
        rates = {"error": str(exc)}
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    sampler = ClockSampler(dev.index)   # every rank samples its own GPU
    sampler.start()
    fs.fs_timing_read()
    fs.fs_timing_enable(True)
    l0 = fs.fs_launch_count()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for s in range(args.steps):
        flush.fill_(float(s))
        ev[s][0].record(stream)
        step()
        ev[s][1].record(stream)
    torch.cuda.synchronize()
    launches = fs.fs_launch_count() - l0
    fs.fs_timing_enable(False)
    (half_ms, apply_ms, prep_ms), (half_n, apply_n, prep_n) = fs.fs_timing_read()
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, dev if world > 1 else None)
    iters, pairs = _work(w, n, m, d)
    value = aggregate_rate(world, pairs, args.steps, total_ms)
    iters_per_s = aggregate_rate(world, iters, args.steps, total_ms)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tensor_path = (path == "tensor") or (path == "auto" and d > 16)
    roof = _dense_roofline(w, path, half_ms, half_n, rates, clocks, sms)

    line = {"metric": METRIC, "value": value, "unit": "score-pairs/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16xf16->f32" if tensor_path else "f32", "data": "synthetic",
            "config": arm_config(w),
            "iters_per_s": iters_per_s, "roofline": roof, "gpu_launches": int(launches),
            "clocks": clocks,
            "apply_ms": apply_ms / max(apply_n, 1) if apply_n else None,
            # preparation (centring, norms, operand packing/tiling) per solve call,
            # included in ms_per_step; and the device workspace the calls use
            "prep_ms_per_step": prep_ms / args.steps,
            "workspace_bytes": int(max(fs.fs_workspace_bytes(n, m, d, 0, path=path),
                                       fs.fs_workspace_bytes(n, m, d, k_out, path=path)
                                       if w.apply else 0))}

    if world == 1 and w.name == DEFAULT_WORKLOAD and not args.no_points:
        line["metric_points"] = {w.name: {
            "workload": w.name, "n": n, "m": m, "d": d, "value": line["value"],
            "unit": "score-pairs/s", "iters_per_s": line["iters_per_s"],
            "ms_per_step": line["ms_per_step"],
            "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                               "frac_of_burst", "traffic", "avg_launch_ms",
                                               "launches") if k in roof},
            "note": "the main measurement of this line"}}
        for name in METRIC_POINTS:
            line["metric_points"][name] = _metric_point(fs, name, dev, rates, path)

    # end to end through the C ABI with pinned host buffers
    if not args.no_e2e:
        host = {k: torch.from_numpy(v).pin_memory() for k, v in inp.items()}
        host["f"] = torch.empty(n).pin_memory()
        host["g0"] = torch.zeros(m).pin_memory()
        host["out"] = torch.empty(n, k_out).pin_memory() if w.apply else None
        estep = _step_fn(fs, w, host, path)
        estep(host)
        torch.cuda.synchronize()
        e2e_ms = []
        for s in range(max(1, min(args.steps, 10))):
            host["g0"].zero_()
            flush.fill_(float(s))
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            estep(host)
            torch.cuda.synchronize()
            e2e_ms.append(1e3 * (time.perf_counter() - t0))
        # bytes the library copies per step: every call stages its host inputs
        fb = 4
        per_solve_h2d = fb * (n * d + n + m * d + m + m)
        per_solve_d2h = fb * (n + m)
        n_solves = len(w.stages)
        h2d = n_solves * per_solve_h2d
        d2h = n_solves * per_solve_d2h
        if w.apply:
            h2d += fb * (n * d + n + m * d + m + n + m + (m * w.k if w.apply == "pv" else 0))
            d2h += fb * n * k_out
        e2e_total = max_over_ranks(sum(e2e_ms), dev if world > 1 else None)
        line["e2e"] = {"value": aggregate_rate(world, pairs, len(e2e_ms), e2e_total),
                       "unit": "score-pairs/s", "h2d_bytes_per_step": int(h2d),
                       "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_total / len(e2e_ms),
                       "timer": "host wall clock around the C-ABI calls, stream synchronised"}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(w, inp, args.cpu_seconds)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_sparse(args, w):
    """The block-sparse solver (workloads with tau > 0): one step is one
    fs_sparse_solve call from a cold start -- Morton sort, centroid stage,
    the workload's block-sparse iterations and the final residual pass."""
    import torch
    from streaming_sinkhorn_solver_gb300 import binding as fs

    rank, world, local = _rank_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    fs.load_library()
    n, m, d = w.n, w.m, w.d
    eps, iters = w.stages[0]
    inp = make_inputs(w.name, seed=replica_seed(w, rank))
    t = {k: torch.from_numpy(v).to(dev) for k, v in inp.items()}
    t["f"] = torch.empty(n, device=dev)
    t["g"] = torch.empty(m, device=dev)
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)  # 256 MB > L2
    kw = dict(coarse_iters=w.coarse_iters, max_iters=iters, tau=w.tau)

    def step(src):
        return fs.fs_sparse_solve(src["X"], src["a"], src["Y"], src["b"], eps, f=src["f"],
                                  g=src["g"], **kw)[2]

    try:
        rates = fs.fs_unit_rates()
    except Exception as exc:  # pragma: no cover
        rates = {"error": str(exc)}
    for _ in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(dev.index)
    sampler.start()
    fs.fs_timing_read()
    fs.fs_timing_enable(True)
    l0 = fs.fs_launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    reps = []
    for s_ in range(args.steps):
        flush.fill_(float(s_))
        ev[s_][0].record(stream)
        reps.append(step(t))
        ev[s_][1].record(stream)
    torch.cuda.synchronize()
    launches = fs.fs_launch_count() - l0
    fs.fs_timing_enable(False)
    (half_ms, _, prep_ms), (half_n, _, _) = fs.fs_timing_read()
    clocks = sampler.stop()
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), dev if world > 1 else None)
    rep = reps[-1]
    dense_pairs = 2 * n * m * iters                     # pairs a dense solve would evaluate
    value = aggregate_rate(world, dense_pairs, args.steps, total_ms)
    kept_per_step = rep["kept_pairs"]
    # the update passes are the timed half-updates; the residual pass is one more
    kept_update = kept_per_step * (2 * rep["iters"]) / max(rep["passes"], 1)
    avg_half_ms = half_ms / max(half_n, 1)
    pairs_per_launch = kept_update / max(2 * rep["iters"], 1)
    peaks = _peaks()
    clk = (clocks or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ex2_clk = rates.get("ex2_per_clk_sm") or EX2_PER_CLK_SM
    fp32_clk = rates.get("fma2_lanes_per_clk_sm") or FP32_LANES_PER_CLK_SM
    rate_src = "measured by fs_unit_rates" if "ex2_per_clk_sm" in rates else "nominal"
    # per kept pair, at the least (reference offsets, as after the first
    # iterations, folded into the column records): d fused multiply-adds and
    # the accumulation -- the same count as the dense FMA path
    fp32_ops = fp32_ops_per_pair(d, False)
    ex2_peak = ex2_clk * sms * clk * 1e6
    fp32_peak = fp32_clk / fp32_ops * sms * clk * 1e6
    alu_peak = min(ex2_peak, fp32_peak)
    achieved = pairs_per_launch / (avg_half_ms * 1e-3)
    roof = {"bound": "alu", "achieved": achieved / 1e9, "peak": alu_peak / 1e9, "unit": "Gpair/s",
            "frac": achieved / alu_peak,
            "peak_source": f"derived: min(MUFU {ex2_clk:.1f} ex2/clk/SM, FP32 {fp32_clk:.1f} "
                           f"lanes/clk/SM / {fp32_ops} lane-ops per kept pair) ({rate_src}) x "
                           f"{sms} SMs x {clk:.0f} MHz (median SM clock in the timed region)",
            "mufu_frac": achieved / ex2_peak, "fp32_frac": achieved / fp32_peak,
            "traffic": _traffic_from_profiles(w.name, "sparse"),
            "kernel": "block_sparse_half_update",
            "avg_launch_ms": avg_half_ms, "launches": half_n,
            "kept_pairs_per_launch": pairs_per_launch,
            "unit_rates": dict(rates, source=rate_src)}
    step_ms = total_ms / args.steps
    line = {"metric": METRIC, "value": value, "unit": "score-pairs/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "value_kind": "dense-equivalent score-pairs/s: 2 n m per iteration over the step "
                          "time; the block-sparse solver evaluates only the kept blocks "
                          "(omitted mass per block below tau of its weight)",
            "config": arm_config(w),
            "iters_per_s": aggregate_rate(world, iters, args.steps, total_ms),
            "kept_pairs_per_s": aggregate_rate(world, kept_per_step, args.steps, total_ms),
            "kept_fraction": kept_per_step / (rep["passes"] * n * m),
            # block pairs the screenings evaluated point by point (one screening per
            # pass when there is no in-loop residual check, as here)
            "exact_bound_fraction": rep["exact_bounds"] / max(
                rep["passes"] * rep["blocks_x"] * rep["blocks_y"], 1),
            # rows whose guarded sum left its range and were recomputed
            "fixed_row_fraction": rep["fixed_rows"] / max(rep["passes"] * (n + m) / 2, 1),
            "residual": rep["residual"], "blocks": [rep["blocks_x"], rep["blocks_y"]],
            "time_split_ms_per_step": {
                "half_updates": half_ms / args.steps, "prep_sort_coarse": prep_ms / args.steps,
                "screening_fixups_and_residual": step_ms - (half_ms + prep_ms) / args.steps},
            "roofline": roof, "gpu_launches": int(launches), "clocks": clocks}
    if not args.no_e2e:
        host = {k: torch.from_numpy(v).pin_memory() for k, v in inp.items()}
        host["f"] = torch.empty(n).pin_memory()
        host["g"] = torch.empty(m).pin_memory()
        step(host)
        e2e = []
        for s_ in range(max(1, min(args.steps, 10))):
            flush.fill_(float(s_))
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            step(host)
            torch.cuda.synchronize()
            e2e.append(1e3 * (time.perf_counter() - t0))
        e2e_total = max_over_ranks(sum(e2e), dev if world > 1 else None)
        line["e2e"] = {"value": aggregate_rate(world, dense_pairs, len(e2e), e2e_total),
                       "unit": "score-pairs/s",
                       "h2d_bytes_per_step": int(4 * (n * d + n + m * d + m + n + m)),
                       "d2h_bytes_per_step": int(4 * (n + m)), "ms_per_step": e2e_total / len(e2e),
                       "timer": "host wall clock around the C-ABI call, stream synchronised"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(w, inp, args.cpu_seconds)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=os.environ.get("FS_BENCH_WORKLOAD", DEFAULT_WORKLOAD),
                    choices=sorted(WORKLOADS))
    ap.add_argument("--path", choices=["auto", "fma", "tensor"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-points", action="store_true",
                    help="skip the other workloads' points after the default workload")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-rows", type=int, default=64)
    args = ap.parse_args()
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    elif w.tau > 0:
        run_sparse(args, w)
    else:
        run_gb300(args, w)


if __name__ == "__main__":
    main()
