#!/usr/bin/env python3
"""Benchmark of the fused hidden-state projection on GB300.

Default workload (one JSON line on rank 0): the wq_a ++ wkv projection of
TensorRT-LLM PR #20636 (DeepSeek-V4.1), X[8, 5120] bf16 times W_cat[1792, 5120]
bf16, outputs [8, 1280] and [8, 512], fused call.

A step is one CUDA-graph replay of --calls fused calls that cycle through C
distinct (W_cat, X, outputs) copies whose weights together exceed three times
the L2 size, so every call streams its weights from HBM.  value = microseconds
per call (lower is better); the roofline object reports the algorithmic bytes
N*K*w + M*K*x + M*N*y of one call divided by that time, against the measured
copy bandwidth in MEASURED_PEAKS.json.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --sweep      # every workload and token count, fused / separate /
                               # PDL off / cuBLAS per split; one JSON line each
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (% of GB300 peak) at M=1/8/64, weights past L2"
DEFAULT_WORKLOAD = ("wq_a_wkv", 8)


# ---------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# The device-code files of each kernel family: its header, its instances and the
# headers it includes.  A profile's DRAM counters stay valid while these are unchanged.
# a kernel's device sources: its header, its instance files and the headers they include
KERNEL_FILES = {
    "reg": ["reg_kernel.cuh", "kernels_reg.cu", "norm_epilogue.cuh"],
    "gemv": ["gemv_kernel.cuh", "kernels_gemv.cu"],
    "stream": ["stream_kernel.cuh", "launch_impl.cuh", "kernels_bf16.cu", "kernels_tf32.cu", "kernels_fp32.cu",
               "norm_epilogue.cuh"],
    "umma": ["umma_kernel.cuh", "kernels_umma.cu"],
}
SHARED_FILES = ["ptx.cuh", "scatter.cuh", "prefetch.cuh", "stream_args.h"]


def strip_comments(src: str) -> str:
    """C/C++ source without // and /* */ comments, blank lines and runs of blanks (string
    literals kept as they are)."""
    import re
    tok = re.compile(r'"(?:\\.|[^"\\])*"|//[^\n]*|/\*.*?\*/', re.S)
    code = tok.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", src)
    out = []
    for ln in code.splitlines():
        parts = re.split(r'("(?:\\.|[^"\\])*")', ln)   # odd items are string literals
        ln = "".join(p if i % 2 else re.sub(r"[ \t]+", " ", p) for i, p in enumerate(parts)).strip()
        if ln:
            out.append(ln)
    return "\n".join(out)


def kernel_sources_sha16(kernel: str) -> str:
    """Hash of a kernel's device sources (its header, its instances and the headers they
    include), comments left out: a comment edit does not void a profile."""
    import hashlib
    csrc = os.path.join(ROOT, "hidden_state_projection_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_FILES[kernel] + SHARED_FILES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(name, M):
    """DRAM bytes per launch from the committed ncu summary of this workload, if that
    summary was taken on the current kernel sources; else None."""
    import glob
    paths = glob.glob(os.path.join(ROOT, "profiles", f"hsp_*_kernel_{name}_m{M}.md"))
    if not paths:
        return None
    path = paths[0]
    kernel = os.path.basename(path).split("_")[1]          # hsp_<kernel>_kernel_<workload>_m<M>.md
    if kernel not in KERNEL_FILES:
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith(("#", "|", " ")):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("kernel_sources_sha256_16") != kernel_sources_sha16(kernel):
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- multi-rank (replicas)

def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the slowest replica sets the job's time).  The
    tensor lives on `device`: CUDA under NCCL, the CPU under gloo."""
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(ms_per_step: float, calls_per_rank: int, world_size: int) -> float:
    """Whole-job µs per call: world_size replicas each ran calls_per_rank calls inside one
    step of ms_per_step (the max over ranks), so the job finished world_size * calls_per_rank
    calls in that time (weak scaling: per-GPU work fixed as N grows)."""
    return ms_per_step * 1000.0 / (calls_per_rank * world_size)


# ---------------------------------------------------------------- the workload's config

def workload_config(wl, M: int, tf32: bool, ws: int) -> dict:
    """The `config` object of both arms: what is computed, not how it is timed."""
    dt = wl.dtype + ("/tf32" if tf32 else "")
    return {
        "workload": f"{wl.name}: X[{M},{wl.K}] {dt} . W_cat[{wl.n_total},{wl.K}]^T, splits "
                    f"{list(wl.splits)} ({'+'.join(wl.split_names)}), fused call",
        "M": M, "K": wl.K, "n_total": wl.n_total, "splits": list(wl.splits),
        "l2_policy": "at least 16 distinct weight copies cycled per call, together more than 3x L2",
        "parallelism": f"replicas x{ws}",
    }


# The metric's token counts beside the headline (wq_a++wkv at M = 8): the configs that
# quote M = 1 and M = 64, and the others at the ends of their token ranges.
PER_M = (("wq_a_wkv_m1", 1, False), ("wq_a_wkv", 8, False), ("qk_indexer", 64, False))
MORE_CONFIGS = (("qk_indexer", 1, False), ("glm_fused_a", 1, False), ("glm_fused_a", 8, False),
                ("indexer_fp32", 64, False), ("indexer_fp32", 64, True), ("indexer_fp32", 16, False))


# ---------------------------------------------------------------- our arm

class Setup:
    """C copies of (x, w_cat, outs) on the device for one workload / M."""

    def __init__(self, wl, M, device, copies=None, tf32=False):
        self.wl, self.M, self.tf32 = wl, M, tf32
        l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20)
        wb = wl.weight_bytes()
        self.copies = copies or max(16, math.ceil(3 * l2 / wb))
        # every copy has its own weights; seeds differ per copy
        base = W.weight_cat(wl, 0).to(device)
        self.w = [base]
        for c in range(1, self.copies):
            # distinct bytes per copy without drawing 16+ full matrices on the host
            self.w.append(torch.roll(base, shifts=c, dims=1).contiguous())
        self.x = [W.activation(wl, M, c % 4).to(device) for c in range(self.copies)]
        dt = self.x[0].dtype
        self.outs = [[torch.empty((M, n), dtype=dt, device=device) for n in wl.splits]
                     for _ in range(self.copies)]

    def bytes_per_call(self):
        return self.wl.algorithmic_bytes(self.M)


def capture_graph(hsp, st: Setup, calls: int, separate=False, prefetch_next=False):
    """Graph of `calls` calls cycling the copies.  prefetch_next: each call also
    prefetches the weights of the next call into L2 (proj_fused_gemm_prefetch)."""
    def one(c):
        if separate:
            hsp.separate_gemm(st.x[c], st.w[c], st.wl.splits, outs=st.outs[c], tf32=st.tf32)
        elif prefetch_next:
            hsp.fused_gemm_prefetch(st.x[c], st.w[c], st.wl.splits, [st.w[(c + 1) % st.copies]],
                                    outs=st.outs[c], tf32=st.tf32)
        else:
            hsp.fused_gemm(st.x[c], st.w[c], st.wl.splits, outs=st.outs[c], tf32=st.tf32)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for c in range(st.copies):  # warm-up outside capture (tensor maps, attributes)
            one(c)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(calls):
            one(i % st.copies)
    return g


def time_graph(g, steps, warmup, barrier=None):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    per = []
    e0.record(stream)
    for _ in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        per.append((a, b))
    e1.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    total = e0.elapsed_time(e1)
    return total, [a.elapsed_time(b) for a, b in per]


def time_e2e(hsp, st: Setup, calls: int):
    """Public API with host buffers: every step copies its tokens from pinned host memory
    to the device, runs the fused projection and returns the outputs to pinned host memory
    (proj_fused_gemm_host through a bound HostCall: one foreign call per step; a staging
    kernel reads the tokens from the mapped host buffer and the projection kernel stores
    the outputs straight into the mapped host buffers), cycling the weight copies as the
    kernel-only timing does.  Also timed: the same steps as recorded host plans
    (proj_host_plan_launch, one graph launch per step)."""
    dev = st.x[0].device
    xh = [st.x[c].cpu().pin_memory() for c in range(4)]
    oh = [torch.empty((st.M, n), dtype=st.x[0].dtype).pin_memory() for n in st.wl.splits]
    xd = torch.empty_like(st.x[0])
    stream = torch.cuda.current_stream()

    def timed(steps):
        for i in range(2 * st.copies):
            steps[i % st.copies]()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(calls):
            steps[i % st.copies]()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / calls

    bound = [hsp.HostCall(xh[c % 4], st.w[c], st.wl.splits, oh, xd, st.outs[c], tf32=st.tf32, stream=stream)
             for c in range(st.copies)]
    us = timed(bound)
    # The same step with the host waiting for each result before the next step (the
    # latency a caller sees when step i + 1 needs step i's outputs): host wall clock.
    n_sync = max(50, min(500, calls // 4))
    for i in range(st.copies):
        bound[i]()
    stream.synchronize()
    t0 = time.perf_counter()
    for i in range(n_sync):
        bound[i % st.copies]()
        stream.synchronize()
    sync_us = (time.perf_counter() - t0) * 1e6 / n_sync
    plans = [hsp.HostPlan(xh[c % 4], st.w[c], st.wl.splits, oh, xd, st.outs[c], tf32=st.tf32, stream=stream)
             for c in range(st.copies)]
    plan_us = timed(plans)
    for p in plans:
        p.close()
    h2d = st.x[0].numel() * st.x[0].element_size()
    d2h = sum(o.numel() * o.element_size() for o in oh)
    del dev
    return us, h2d, d2h, plan_us, sync_us


def cpu_baseline(wl, M, budget_s=12.0):
    import oracle
    oracle.build()
    cores = oracle.cpu_count()
    x = W.to_numpy_bits(W.activation(wl, M))
    w = W.to_numpy_bits(W.weight_cat(wl))
    dt = oracle.BF16 if wl.dtype == "bf16" else oracle.FP32
    oracle.fused(x, w, wl.splits, dt, threads=cores)  # warm-up
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.fused(x, w, wl.splits, dt, threads=cores)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 200:
            break
    return {"value": el * 1e6 / n, "unit": "µs/call", "cores": cores, "kind": "oracle",
            "sample": f"{n} full calls of {wl.name} M={M} (fp64 oracle, {cores} threads, "
                      f"{oracle.host_description()})"}


def time_rmsnorm_variants(hsp, dev, calls, steps, warmup):
    """µs per call of the RMSNorm-epilogue call at wq_a++wkv M = 8 (q_norm / kv_norm on
    both splits), with a caller workspace and with the library's fixed array (one kernel
    per call either way: every call leaves the arrival counters at zero), same rotation
    as above."""
    wl, M, cols = W.WORKLOADS["wq_a_wkv"], 8, (1280, 512)
    st = Setup(wl, M, dev)
    g0 = torch.Generator().manual_seed(3)
    gam = [(1.0 + 0.1 * torch.randn(c, generator=g0)).to(torch.bfloat16).to(dev) for c in cols]
    ws_t = torch.zeros(hsp.rmsnorm_workspace_bytes(M, wl.K, wl.splits, cols), dtype=torch.uint8, device=dev)
    res = {}
    for label, static in (("caller_workspace_us", False), ("static_workspace_us", True)):
        def one(c):
            if static:
                hsp.fused_gemm_rmsnorm_static(st.x[c], st.w[c], wl.splits, cols, gam, 1e-6, outs=st.outs[c])
            else:
                hsp.fused_gemm_rmsnorm(st.x[c], st.w[c], wl.splits, cols, gam, 1e-6, ws_t, outs=st.outs[c])
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for c in range(st.copies):
                one(c)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(calls):
                one(i % st.copies)
        tot, _ = time_graph(g, steps, warmup)
        res[label] = round(tot * 1000.0 / (steps * calls), 4)
        del g
    res["how"] = ("proj_fused_gemm_rmsnorm (caller workspace) and proj_fused_gemm_rmsnorm_static (the library's "
                  "built-in array, one kernel per call) at wq_a++wkv M=8, q_norm / kv_norm on both splits")
    del st
    torch.cuda.empty_cache()
    return res


def time_config(hsp, wl, M, tf32, dev, calls, steps, warmup, barrier, ws):
    """µs per call and the HBM roofline of one more config, timed like the headline."""
    st = Setup(wl, M, dev, tf32=tf32)
    g = capture_graph(hsp, st, calls)
    total_ms, _ = time_graph(g, steps, warmup, barrier)
    del g
    ms_step = max_over_ranks(total_ms / steps, dev) if ws > 1 else total_ms / steps
    us_gpu = ms_step * 1000.0 / calls
    peak, _ = measured_peaks()
    b = st.bytes_per_call()
    achieved = b / (us_gpu * 1e-6) / 1e9
    kernel = hsp.describe_plan(M, wl.K, wl.n_total, hsp.PROJ_TF32 if tf32 else
                               (hsp.PROJ_BF16 if wl.dtype == "bf16" else hsp.PROJ_FP32))["engine"]
    out = {"us_per_call": round(job_us_per_call(ms_step, calls, ws), 4), "bytes_per_call": b,
           "gpu_launches": steps * calls,
           "achieved_gbs": round(achieved, 1), "frac": round(achieved / peak, 4),
           "engine": ENGINE_NAMES.get(kernel, str(kernel)), "weight_copies": st.copies,
           "traffic": profiled_traffic(wl.name, M) if not tf32 else None,
           "config": workload_config(wl, M, tf32, ws)}
    del st
    torch.cuda.empty_cache()
    return out


ENGINE_NAMES = {0: "streaming", 1: "tcgen05", 2: "register ring", 3: "fp32 register GEMV"}


def run_ours(args):
    ws, rank, local = dist_env()
    import hidden_state_projection_gb300 as hsp
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    barrier = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        barrier = dist.barrier
    hsp.lib()
    hsp.set_options(pdl=not args.no_pdl)
    name, M = args.workload, args.M
    wl = W.WORKLOADS[name]
    st = Setup(wl, M, dev, tf32=args.tf32)
    g = capture_graph(hsp, st, args.calls)
    with ClockSampler(local) as clk:
        total_ms, per = time_graph(g, args.steps, args.warmup, barrier)
        del g
        hsp.check_device_error()
        # the metric's other token counts, same rotation, graph length and clocks
        per_m, more = {}, {}
        if not args.headline_only:
            for dest, table in ((per_m, PER_M), (more, MORE_CONFIGS)):
                for wname, m, tf in table:
                    if (wname, m, tf) == (name, M, args.tf32):
                        continue
                    dest[f"{wname} M={m}{' tf32' if tf else ''}"] = time_config(
                        hsp, W.WORKLOADS[wname], m, tf, dev, args.calls, max(3, args.steps // 2), args.warmup,
                        barrier, ws)
        rms = None
        if not args.headline_only and ws == 1:
            rms = time_rmsnorm_variants(hsp, dev, args.calls, max(3, args.steps // 2), args.warmup)
    hsp.check_device_error()
    ms_per_step = max_over_ranks(total_ms / args.steps, dev) if ws > 1 else total_ms / args.steps
    # whole job: every rank ran args.calls calls per step, all within ms_per_step
    us_call = job_us_per_call(ms_per_step, args.calls, ws)
    bytes_call = st.bytes_per_call()
    # roofline of one GPU's kernel: its own calls in the (max over ranks) step time
    achieved = bytes_call / (ms_per_step * 1000.0 / args.calls * 1e-6) / 1e9
    peak, peak_kind = measured_peaks()
    e2e_us, h2d, d2h, e2e_plan_us, e2e_sync_us = time_e2e(hsp, st, args.e2e_calls)
    # Same calls, each also prefetching the next call's weights into L2 (the cross-kernel
    # weight prefetch of the GLM fused-A kernel): reported beside the headline, not as it.
    gp = capture_graph(hsp, st, args.calls, prefetch_next=True)
    tot_pf, _ = time_graph(gp, max(3, args.steps // 2), args.warmup, barrier)
    us_pf = tot_pf * 1000.0 / (max(3, args.steps // 2) * args.calls)
    del gp
    # Same calls with the dependent launch triggered at kernel entry: the order the pages'
    # tinygemm2 uses (valid only when every PDL dependent waits on its grid dependency, as
    # these calls do).  Reported beside the headline; the library's default stays after the
    # stores.
    hsp.set_options(trigger_early=True)
    ge = capture_graph(hsp, st, args.calls)
    hsp.set_options(trigger_early=False)
    tot_early, _ = time_graph(ge, max(3, args.steps // 2), args.warmup, barrier)
    us_early = tot_early * 1000.0 / (max(3, args.steps // 2) * args.calls)
    del ge
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(us_call, 4),
        "unit": "µs/call",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else ("tf32" if args.tf32 else "f32"),
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights; shapes of the pages' projections)",
        "config": workload_config(wl, M, args.tf32, ws),
        "timing": {"calls_per_step": args.calls, "weight_copies": st.copies,
                   "weight_bytes_cycled": st.copies * wl.weight_bytes(),
                   "how": "CUDA-graph replay of calls_per_step calls per step, CUDA events on the "
                          "launching stream; weights past L2 by rotation (inputs larger than L2)",
                   "pdl": not args.no_pdl},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": args.traffic if args.traffic is not None else profiled_traffic(name, M),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "bytes_per_call": bytes_call, "us_per_call_per_gpu": round(ms_per_step * 1000.0 / args.calls, 4)},
        "e2e": {"value": round(e2e_us, 3), "unit": "µs/call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "public API proj_fused_gemm_host per step (bound HostCall): x read from pinned host memory by the token staging kernel, fused call (PDL-chained), outputs stored by the kernel into pinned mapped host memory",
                "host_plan_us": round(e2e_plan_us, 3),
                "synchronous_step_us": round(e2e_sync_us, 3)},
        "gpu_launches": args.steps * args.calls,   # one fused kernel per call, all inside the graph
        "with_l2_prefetch_of_next_weights": {
            "us_per_call": round(us_pf, 4), "gbs": round(bytes_call / (us_pf * 1e-6) / 1e9, 1),
            "how": "proj_fused_gemm_prefetch: call i also prefetches call i+1's W_cat into L2 "
                   "(every weight still comes from HBM once per call; not the headline)"},
        "with_trigger_at_entry": {
            "us_per_call": round(us_early, 4), "gbs": round(bytes_call / (us_early * 1e-6) / 1e9, 1),
            "how": "trigger_early option: each call lets the next launch at its entry (tinygemm2's "
                   "order; the next call still waits on its grid dependency before reading tokens); "
                   "not the headline, the default triggers after the output stores"},
        "clocks": clocks,
        "step_ms_min": round(min(per), 5), "step_ms_median": round(statistics.median(per), 5),
    }
    if per_m:
        headline = {"us_per_call": line["value"], "bytes_per_call": bytes_call, "achieved_gbs": round(achieved, 1),
                    "frac": round(achieved / peak, 4), "headline": True}
        line["per_M"] = {f"{name} M={M}{' tf32' if args.tf32 else ''}": headline, **per_m}
        line["more_configs"] = more
    if rms:
        line["rmsnorm_epilogue"] = rms

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, M, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = W.WORKLOADS[args.workload]
    M = args.M
    cores = oracle.cpu_count()
    x = W.to_numpy_bits(W.activation(wl, M))
    w = W.to_numpy_bits(W.weight_cat(wl))
    dt = oracle.BF16 if wl.dtype == "bf16" else oracle.FP32
    for _ in range(args.warmup):
        oracle.fused(x, w, wl.splits, dt, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.fused(x, w, wl.splits, dt, threads=cores)
    el = time.perf_counter() - t0
    us = el * 1e6 / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 2), "unit": "µs/call",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1000, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights; shapes of the pages' projections)",
        "config": workload_config(wl, M, args.tf32, ws),
        "cpu_baseline": {"value": round(us, 2), "unit": "µs/call", "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} full calls (one per step) on {cores} threads, {oracle.host_description()}"},
        "e2e": {"value": round(us, 2), "unit": "µs/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- sweep

def run_sweep(args):
    import torch.nn.functional as F
    import hidden_state_projection_gb300 as hsp
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hsp.lib()
    peak, _ = measured_peaks()
    for name, wl in W.WORKLOADS.items():
        modes = [False, True] if wl.dtype == "fp32" else [False]
        for M in wl.Ms:
            for tf32 in modes:
                st = Setup(wl, M, dev, tf32=tf32)
                res = {"workload": name, "M": M, "dtype": wl.dtype + ("/tf32" if tf32 else ""),
                       "bytes": st.bytes_per_call()}
                for label, sep, pdl, pf, early in (
                        ("fused", False, True, False, False), ("separate", True, True, False, False),
                        ("fused_nopdl", False, False, False, False), ("fused_prefetch_next", False, True, True, False),
                        ("fused_trigger_at_entry", False, True, False, True)):
                    hsp.set_options(pdl=pdl, trigger_early=early)
                    g = capture_graph(hsp, st, args.calls, separate=sep, prefetch_next=pf)
                    hsp.set_options(trigger_early=False)
                    tot, _ = time_graph(g, args.steps, args.warmup)
                    us = tot * 1000.0 / (args.steps * args.calls)
                    res[label + "_us"] = round(us, 3)
                    res[label + "_gbs"] = round(st.bytes_per_call() / us / 1e3, 1)
                    del g
                hsp.set_options(pdl=True)
                # cuBLAS (torch.nn.functional.linear) per split, same rotation
                views = [[w[o:o + n] for o, n in zip([sum(wl.splits[:i]) for i in range(len(wl.splits))],
                                                      wl.splits)] for w in st.w]
                torch.backends.cuda.matmul.allow_tf32 = tf32
                for c in range(st.copies):
                    for v in views[c]:
                        F.linear(st.x[c], v)
                torch.cuda.synchronize()
                gg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gg):
                    for i in range(args.calls):
                        c = i % st.copies
                        for v in views[c]:
                            F.linear(st.x[c], v)
                tot, _ = time_graph(gg, args.steps, args.warmup)
                us = tot * 1000.0 / (args.steps * args.calls)
                res["cublas_split_us"] = round(us, 3)
                res["fused_frac_of_peak"] = round(res["fused_gbs"] / peak, 4)
                print(json.dumps(res), flush=True)
                del gg, st
                torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD[0], choices=list(W.WORKLOADS))
    ap.add_argument("--M", type=int, default=DEFAULT_WORKLOAD[1])
    ap.add_argument("--tf32", action="store_true")
    ap.add_argument("--calls", type=int, default=1000, help="fused calls per step (graph replay)")
    ap.add_argument("--e2e-calls", type=int, default=2000)
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of this kernel (reported as is)")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the headline workload only (no per_M / more_configs entries)")
    args = ap.parse_args()
    if args.steps < 1 or args.warmup < 0:
        ap.error("--steps >= 1 and --warmup >= 0")
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
