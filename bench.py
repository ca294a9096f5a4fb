"""Benchmark: exact per-row bf16 top-k on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--plan P] [--dtype bf16|f16|f32] [--k K]

A step is one call of the whole path (load, key encode, span select, span
merge, write) over one batch: the 256 x 248320 bf16 draft window with k = 20
(16 streams x a 16-row draft window of a 248320-column vocabulary).  Inputs
are resident in HBM before the timed region; the timed loop rotates over
enough input copies that each call reads DRAM, not L2.  With N > 1 (torchrun,
one process per GPU) every rank runs its own batch (weak scaling: rows are
independent, there is no data-path exchange); the barrier-bracketed time is
the max over ranks.

``--impl reference`` times the CPU oracle (all host cores) on the same
workload instead -- the reference arm; under torchrun only rank 0 runs it.

``--dtype`` / ``--k`` time tf_topk_select on the same values in another
format (fp32: the bf16 values widened exactly; fp16: rounded to nearest) or
with another k; ``--plan 64`` forces its wide kernel.  The defaults are the
bf16, k = 20 call above.
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
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "rows/s and µs/call for bf16 row top-k; achieved HBM GB/s vs GB300 peak"
DEFAULT_WORKLOAD = "256x248320_k20"
CSRC = ROOT / "wide_bf16_row_gb300" / "csrc"
KERNEL_SOURCE = CSRC / "tf_topk.cu"
# the source file each profiled kernel is built from (its hash dates a profile)
KERNEL_FILES = {"topk_f32_cluster_kernel": CSRC / "tf_topk_f32.cu"}
PROFILES = ROOT / "profiles"
# the kernel each launch plan runs (the ncu summaries are named after it)
PLAN_KERNEL = {1: "topk_cluster_kernel_S1", 2: "topk_cluster_kernel_S2", 4: "topk_cluster_kernel_S4",
               8: "topk_cluster_kernel_S8", 16: "topk_cluster_kernel_S16", 32: "topk_stream_kernel",
               64: "topk_wide_kernel"}
PLAN_NAME = {1: "single", 2: "cluster2", 4: "cluster4", 8: "cluster8", 16: "cluster16", 32: "stream", 64: "wide"}
# logit formats of tf_topk_select: (TF_TOPK_DTYPE_* code, bit-pattern type)
FORMATS = {"bf16": (0, np.uint16), "f16": (1, np.uint16), "f32": (2, np.uint32)}
FAST_MAX_K = 64
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- helpers

def dist_env() -> tuple[int, int, int]:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, steps: int, world: int, max_elapsed_s: float) -> float:
    """Units all ranks processed / the slowest rank's time."""
    return units_per_rank * steps * world / max_elapsed_s


def measured_peak_hbm() -> tuple[float, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(kernel: str = "") -> str:
    return hashlib.sha256(KERNEL_FILES.get(kernel, KERNEL_SOURCE).read_bytes()).hexdigest()


def profiled_traffic(kernel: str, workload: str) -> int | None:
    """DRAM bytes per launch of `kernel` on this workload, from the committed
    ncu summary, if it was taken on the kernel's current source (else None)."""
    try:
        text = (PROFILES / f"{kernel}_{workload}.md").read_text()
    except OSError:
        return None
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    if not h or not t or h.group(1) != kernel_source_hash(kernel):
        return None
    return int(t.group(1))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples, kept with their wall time."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 20):
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout: float = 10.0):
        t = time.time()
        while self.proc and not self.samples and time.time() - t < timeout:
            time.sleep(0.01)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        note = "sampled inside the timed region"
        if not inside and self.samples:
            # the region is shorter than the sampling period: take the nearest samples
            near = sorted(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))[:2]
            inside = [s for _, s in near]
            note = "timed region shorter than the sampling period: nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[0]) for s in inside if num(s[0]) is not None]
        smax = [num(s[1]) for s in inside if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def nvsmi_id(dev) -> str:
    """nvidia-smi's id for a torch device: its PCI address when torch knows it."""
    import torch

    p = torch.cuda.get_device_properties(dev)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return str(dev.index or 0)


def make_workload(name: str, rank: int = 0):
    from wide_bf16_row_gb300 import synth

    if name not in synth.NAMED:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(synth.NAMED)}")
    return synth.NAMED[name]()


def format_bits(w, fmt: str) -> np.ndarray:
    """The workload's values as bit patterns of `fmt`: bf16 as drawn, fp32
    widened exactly, fp16 rounded to nearest."""
    if fmt == "bf16":
        return w.logits
    from wide_bf16_row_gb300 import synth

    vals = synth.bf16_to_float(w.logits)
    if fmt == "f32":
        return np.ascontiguousarray(vals).view(np.uint32)
    with np.errstate(over="ignore", invalid="ignore"):
        return vals.astype(np.float16).view(np.uint16)


def run_label(w, fmt: str, k: int) -> str:
    """The workload's name, with the format and k when they are not its own."""
    return w.name if (fmt == "bf16" and k == w.k) else f"{w.rows}x{w.cols}_k{k}_{fmt}"


def workload_config(w, extra: dict | None = None) -> dict:
    cfg = {"workload": w.name, "rows": w.rows, "cols": w.cols, "k": w.k,
           "row_stride": w.row_stride}
    if extra:
        cfg.update(extra)
    return cfg


def isolated_launches(step, stream, dev, n: int) -> list[float]:
    """n launches, each alone between its own pair of events (synchronised
    before and after, so none overlaps a neighbour); ms per launch."""
    import torch

    out = []
    for i in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        a.record(stream)
        step(i)
        b.record(stream)
        torch.cuda.synchronize(dev)
        out.append(a.elapsed_time(b))
    return out


# The workloads the per-config table covers: the four named ones, the widest
# of them with a -inf mask, and sweep points.
PER_CONFIG = (
    ("1x4096_k8", None),
    ("15x98592_k16", None),
    ("16x248320_k64_specials", None),
    ("256x248320_k20", None),
    ("256x248320_k20_masked", None),
    ("sweep_1024x248320_k20", (248320, 1024, 20)),
    ("sweep_64x151936_k64", (151936, 64, 64)),
    ("sweep_4x98592_k8", (98592, 4, 8)),
    ("sweep_1024x4096_k20", (4096, 1024, 20)),
)


def per_config_workload(name: str, sweep):
    from wide_bf16_row_gb300 import synth

    if sweep:
        return synth.config_sweep(*sweep)
    return synth.config_masked_window() if name.endswith("_masked") else synth.NAMED[name]()


def measure_config(w, dev, peak: float, cpu: bool, cpu_seconds: float) -> dict:
    """One workload through tf_topk_bf16 (the library's own plan): kernel time
    per call from a CUDA graph of back-to-back calls (no host issue cost),
    inputs rotating over copies that together exceed L2 four times where that
    fits (small inputs stay L2-resident, said in `l2`); the same calls issued
    from Python; single isolated calls; the host cost of one call; and the
    oracle on the host cores."""
    import torch

    from wide_bf16_row_gb300 import topk

    rows, cols, stride, k = w.rows, w.cols, w.row_stride, w.k
    in_bytes = rows * stride * 2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    want = max(2, math.ceil(4 * l2 / in_bytes))
    nbuf = min(want, 64)
    host = torch.from_numpy(w.logits.view(np.int16))
    bufs = [host.to(dev) for _ in range(nbuf)]
    views = [b.as_strided((rows, cols), (stride, 1)) for b in bufs]
    out = (torch.empty((rows, k), dtype=torch.int32, device=dev),
           torch.empty((rows, k), dtype=torch.int16, device=dev),
           torch.empty((rows,), dtype=torch.int32, device=dev),
           torch.empty((rows,), dtype=torch.int32, device=dev))
    plan = topk.plan(rows, cols, k)
    side = torch.cuda.Stream(dev)

    def call(i, s):
        topk.topk_bf16(views[i % nbuf], k, out=out, stream=s)

    with torch.cuda.stream(side):
        for i in range(5):
            call(i, side)
    torch.cuda.synchronize(dev)
    # kernel time: a graph of G back-to-back calls, replayed R times
    n_calls = max(2 * nbuf, 40)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for i in range(n_calls):
            call(i, side)
    reps = max(3, min(200, int(2e5 / max(1.0, n_calls))))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):  # a graph replays on the current stream
        graph.replay()
        torch.cuda.synchronize(dev)
        a.record(side)
        for _ in range(reps):
            graph.replay()
        b.record(side)
    torch.cuda.synchronize(dev)
    us_graph = a.elapsed_time(b) * 1e3 / (reps * n_calls)
    # the same calls issued from Python, back to back
    n_py = 200
    a.record(side)
    for i in range(n_py):
        call(i, side)
    b.record(side)
    torch.cuda.synchronize(dev)
    us_python = a.elapsed_time(b) * 1e3 / n_py
    # host cost of one call (argument checks, plan, launch): no synchronisation
    t0 = time.perf_counter()
    for i in range(n_py):
        call(i, side)
    host_us = (time.perf_counter() - t0) * 1e6 / n_py
    torch.cuda.synchronize(dev)
    iso = [x * 1e3 for x in isolated_launches(lambda i: call(i, side), side, dev, 30)]
    alg = rows * cols * 2 + rows * k * 6 + rows * 8
    gbs = alg / (us_graph * 1e-6) / 1e9
    res = {
        "rows": rows, "cols": cols, "k": k, "row_stride": stride,
        "plan": PLAN_NAME.get(plan, str(plan)),
        "us_per_call": us_graph,
        "rows_per_s": rows / (us_graph * 1e-6),
        "gbs": gbs, "frac_of_peak": gbs / peak,
        "algorithmic_bytes": alg,
        "us_per_call_python_issued": us_python,
        "us_isolated_p10_p50_p90": [round(float(np.percentile(iso, q)), 2) for q in (10, 50, 90)],
        "host_us_per_call": host_us,
        "timing": f"CUDA graph of {n_calls} back-to-back calls, {reps} replays, CUDA events",
        "l2": (f"inputs rotate over {nbuf} device copies ({nbuf * in_bytes / 1e6:.0f} MB)"
               + ("" if nbuf >= want else "; fits L2 (L2-resident)")),
    }
    if cpu:
        all_cores = time_oracle(w, budget_s=cpu_seconds)
        one = time_oracle(w, budget_s=cpu_seconds / 2, rows_per_call=1)
        res["oracle_rows_per_s"] = all_cores["value"]
        res["oracle_cores"] = all_cores["cores"]
        res["oracle_rows_per_s_1core"] = one["value"]
    del bufs, views
    torch.cuda.empty_cache()
    return res


def per_config_table(dev, peak: float, cpu: bool, cpu_seconds: float) -> dict:
    table = {}
    for name, sweep in PER_CONFIG:
        w = per_config_workload(name, sweep)
        table[name] = measure_config(w, dev, peak, cpu, cpu_seconds)
    return table


# The draft heads the fused head-with-top-k entry point is measured on.
HEAD_CONFIGS = (
    ("15x2048x98592_k16", "config_head_draft"),
    ("16x2048x248320_k64", "config_head_wide"),
)


def measure_head(h, dev, peak: float, cpu: bool, cpu_seconds: float) -> dict:
    """One draft head through tf_topk_head_bf16 (the product and the top-k in
    one kernel, plus the merge of the per-CTA lists) and, on the same device,
    the two-step path it replaces: cuBLAS's bf16 product into a logit matrix,
    then tf_topk_bf16.  Each timed as a CUDA graph of back-to-back calls
    (the weight matrix exceeds L2, so every call streams it from HBM)."""
    import torch

    from wide_bf16_row_gb300 import topk

    rows, dim, vocab, k = h.hidden.shape[0], h.hidden.shape[1], h.weight.shape[0], h.k
    hid = torch.from_numpy(h.hidden.view(np.int16)).to(dev).view(torch.bfloat16)
    w = torch.from_numpy(h.weight.view(np.int16)).to(dev).view(torch.bfloat16)
    ws = torch.empty((topk.tf_topk_head_bf16_workspace(rows, k),), dtype=torch.uint8, device=dev)
    out = (torch.empty((rows, k), dtype=torch.int32, device=dev),
           torch.empty((rows, k), dtype=torch.int16, device=dev),
           torch.empty((rows,), dtype=torch.int32, device=dev),
           torch.empty((rows,), dtype=torch.int32, device=dev))
    out2 = tuple(torch.empty_like(t) for t in out)
    logits = torch.empty((rows, vocab), dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream(dev)

    def fused():
        topk.head_topk_bf16(hid, w, k, out=out, workspace=ws, stream=side)

    def two_step():
        torch.matmul(hid, w.t(), out=logits)
        topk.topk_bf16(logits, k, out=out2, stream=side)

    def graph_us(fn, n_calls=20, reps=20):
        with torch.cuda.stream(side):
            for _ in range(3):
                fn()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for _ in range(n_calls):
                fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(side):
            graph.replay()
            torch.cuda.synchronize(dev)
            a.record(side)
            for _ in range(reps):
                graph.replay()
            b.record(side)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) * 1e3 / (reps * n_calls)

    us_fused = graph_us(fused)
    us_two = graph_us(two_step)
    same = all(bool(torch.equal(x, y)) for x, y in zip(out, out2))
    alg = vocab * dim * 2 + rows * dim * 2 + rows * k * 6 + rows * 8
    gbs = alg / (us_fused * 1e-6) / 1e9
    res = {
        "rows": rows, "dim": dim, "vocab": vocab, "k": k,
        "us_per_call": us_fused,
        "us_per_call_cublas_then_topk": us_two,
        "speedup_vs_cublas_then_topk": us_two / us_fused,
        "rows_per_s": rows / (us_fused * 1e-6),
        "gbs": gbs, "frac_of_peak": gbs / peak, "bound": "hbm",
        "algorithmic_bytes": alg,
        "same_result_as_cublas_then_topk": same,
        "timing": "CUDA graph of 20 back-to-back calls, 20 replays, CUDA events; weight > L2",
    }
    if cpu:
        from oracle import head as head_oracle

        n = 1
        head_oracle.topk(h.hidden[:n], h.weight, k)  # warm
        reps, t0 = 0, time.perf_counter()
        while True:
            head_oracle.topk(h.hidden[:n], h.weight, k)
            reps += 1
            if time.perf_counter() - t0 > cpu_seconds / 2:
                break
        res["oracle_rows_per_s"] = reps * n / (time.perf_counter() - t0)
        res["oracle_sample"] = f"{n} row(s) of the head per call, numpy float64 product on the host's BLAS threads"
    del hid, w, ws, logits
    torch.cuda.empty_cache()
    return res


def head_table(dev, peak: float, cpu: bool, cpu_seconds: float) -> dict:
    from wide_bf16_row_gb300 import synth

    return {name: measure_head(getattr(synth, fn)(), dev, peak, cpu, cpu_seconds) for name, fn in HEAD_CONFIGS}


# ----------------------------------------------------------------------------- oracle timing

def time_oracle(w, budget_s: float, rows_per_call: int | None = None, bits: np.ndarray | None = None,
                k: int | None = None, fmt: str = "bf16") -> dict:
    """The CPU oracle (as it stands) on a bounded sample of the workload's rows,
    all host cores; repeated until ``budget_s`` of wall time has passed."""
    import oracle

    cores = host_cores()
    bits = w.logits if bits is None else bits
    k = w.k if k is None else k
    n = min(w.rows, rows_per_call or max(cores, 1))
    sample = bits[:n]
    oracle.topk(sample, w.cols, k, nthreads=cores, dtype=fmt)  # load + warm
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.topk(sample, w.cols, k, nthreads=cores, dtype=fmt)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": n * reps / el, "unit": "rows/s", "cores": min(cores, n), "kind": "oracle",
            "sample": f"first {n} rows of {run_label(w, fmt, k)}, {reps} repetitions, {el:.2f} s wall, "
                      f"{min(cores, n)} threads"}


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle

    w = make_workload(args.workload)
    k = args.k or w.k
    bits = format_bits(w, args.dtype)
    cores = host_cores()
    # one step = the top-k of one row of the batch; `cores` steps run side by side
    per_call = max(1, cores)
    order = np.arange(args.steps + args.warmup) % w.rows
    for s in range(0, args.warmup, per_call):
        rows = order[s: min(args.warmup, s + per_call)]
        oracle.topk(bits[rows], w.cols, k, nthreads=cores, dtype=args.dtype)
    t0 = time.perf_counter()
    done = 0
    while done < args.steps:
        rows = order[args.warmup + done: args.warmup + min(args.steps, done + per_call)]
        oracle.topk(bits[rows], w.cols, k, nthreads=cores, dtype=args.dtype)
        done += len(rows)
    el = time.perf_counter() - t0
    value = args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, {
            **({} if run_label(w, args.dtype, k) == w.name
               else {"workload": run_label(w, args.dtype, k), "k": k, "format": args.dtype}),
            "step": f"top-k of one row; host-core batches of {per_call} rows"}),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": min(cores, per_call),
                         "kind": "oracle",
                         "sample": f"{args.steps} rows of {run_label(w, args.dtype, k)} (cycling), "
                                   f"{per_call} per call"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm

def run_ours(args) -> None:
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from wide_bf16_row_gb300 import topk

    w = make_workload(args.workload, rank)
    rows, cols, stride = w.rows, w.cols, w.row_stride
    k = args.k or w.k
    fmt = args.dtype
    code, _ = FORMATS[fmt]
    bits = format_bits(w, fmt)
    esize = bits.dtype.itemsize
    tint = torch.int32 if esize == 4 else torch.int16
    in_bytes = rows * stride * esize
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nbuf = max(2, math.ceil(4 * l2 / in_bytes))
    host = torch.from_numpy(bits.view(np.int32 if esize == 4 else np.int16))
    bufs = [host.to(dev) for _ in range(nbuf)]
    views = [b.as_strided((rows, cols), (stride, 1)) for b in bufs]
    out = (torch.empty((rows, k), dtype=torch.int32, device=dev),
           torch.empty((rows, k), dtype=tint, device=dev),
           torch.empty((rows,), dtype=torch.int32, device=dev),
           torch.empty((rows,), dtype=torch.int32, device=dev))
    stream = torch.cuda.current_stream(dev)
    plan_arg = args.plan
    # bf16 with k <= 64 runs the tf_topk_bf16 plans, fp16 with k <= 64 their
    # cluster plans (one CTA per row becomes the wide kernel); anything else
    # the wide kernel
    fast = fmt in ("bf16", "f16") and k <= FAST_MAX_K and plan_arg != 64
    plan = (plan_arg if plan_arg else topk.plan(rows, cols, k)) if fast else 64
    if fmt == "f16" and plan == 32:
        plan = 64
    # fp32 with k <= 64 on AUTO: the library's fp32 cluster kernel
    f32_cluster = fmt == "f32" and k <= FAST_MAX_K and plan_arg == 0
    kernel = "topk_f32_cluster_kernel" if f32_cluster else PLAN_KERNEL.get(plan, "")
    label = run_label(w, fmt, k)

    def call(view):
        s = torch.cuda.current_stream(dev)  # the capture stream while a graph is captured
        if fmt == "bf16" and k == w.k and plan_arg != 64:
            topk.topk_bf16(view, k, plan=plan_arg, out=out, stream=s)
        else:
            topk.select_topk(view, k, dtype=code, plan=plan_arg, out=out, stream=s)

    def step(i: int):
        call(views[i % nbuf])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    # the K timed steps, captured once as a CUDA graph (the same launches on
    # the same rotating inputs), so that the timed region holds device work
    # only, not the host's issue of each launch
    graph, inner = None, None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.stream(cap):  # any per-stream scratch is made before the capture
            step(0)
        torch.cuda.synchronize(dev)
        # events recorded by the graph itself, around its K launches: no
        # host issue gap between the start event and the first launch
        try:
            inner = (torch.cuda.Event(enable_timing=True, external=True),
                     torch.cuda.Event(enable_timing=True, external=True))
        except TypeError:
            inner = None
        with torch.cuda.graph(graph, stream=cap):
            if inner:
                inner[0].record(cap)
            for i in range(args.steps):
                step(i)
            if inner:
                inner[1].record(cap)
        graph.replay()  # one untimed replay
        torch.cuda.synchronize(dev)

    # the timed launches run back to back (each may be scheduled while the
    # previous one finishes); isolated launches are timed afterwards, apart
    sampler = ClockSampler(nvsmi_id(dev)) if not args.no_clocks else None
    if sampler:
        sampler.wait_first()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    elapsed_outer_ms = start.elapsed_time(end)
    elapsed_ms = inner[0].elapsed_time(inner[1]) if graph is not None and inner else elapsed_outer_ms
    launch_ms = isolated_launches(step, stream, dev, n=min(50, max(3, args.steps)))

    # L2-warm: the same input every call (draft logits often sit in L2 right
    # after the head that wrote them); reported beside the L2-cold value
    warm_steps = max(1, min(args.steps, 2000))
    for _ in range(3):
        call(views[0])
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(warm_steps):
        call(views[0])
    w1.record(stream)
    torch.cuda.synchronize(dev)
    warm_us = w0.elapsed_time(w1) * 1e3 / warm_steps
    max_ms = max_over_ranks(elapsed_ms, world, dev)
    value = whole_job_rate(rows, args.steps, world, max_ms / 1e3)
    # average launch duration: this rank's timed region over its launches
    avg_launch_s = elapsed_ms / 1e3 / args.steps
    isolated_s = statistics.mean(launch_ms) / 1e3 if launch_ms else None
    alg_bytes = rows * cols * esize + rows * k * (4 + esize) + rows * 8
    peak, peak_kind = measured_peak_hbm()
    achieved = alg_bytes / avg_launch_s / 1e9

    # parity of the timed configuration (all rows) against the CPU oracle? that is
    # the tests' job; here: one cheap self-check that the output is a real result
    idx = out[0].cpu()
    assert int(out[2][0].item()) == min(k, cols) and int(idx[0, 0].item()) >= 0

    # end to end through the public API: pinned host input -> device, top-k, outputs -> host
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    pinned_in = host.pin_memory()
    dbuf = torch.empty_like(bufs[0])
    dview = dbuf.as_strided((rows, cols), (stride, 1))
    h_out = tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in out)
    for _ in range(2):
        dbuf.copy_(pinned_in, non_blocking=True)
        call(dview)
        for h, d in zip(h_out, out):
            h.copy_(d, non_blocking=True)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        dbuf.copy_(pinned_in, non_blocking=True)
        call(dview)
        for h, d in zip(h_out, out):
            h.copy_(d, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = whole_job_rate(rows, e2e_steps, world, e2e_ms / 1e3)
    h2d = rows * stride * esize
    d2h = rows * k * 4 + rows * k * esize + rows * 4 + rows * 4

    per_config = None
    head = None
    tables = "none" if args.no_per_config else args.tables
    if rank == 0 and world == 1 and tables == "all":
        per_config = per_config_table(dev, peak, not args.no_cpu_baseline, min(0.6, args.cpu_seconds))
    if rank == 0 and world == 1 and tables in ("all", "head"):
        head = head_table(dev, peak, not args.no_cpu_baseline, min(0.6, args.cpu_seconds))

    cpu = None
    cpu_1core = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(w, budget_s=args.cpu_seconds, bits=bits, k=k, fmt=fmt)
        cpu_1core = time_oracle(w, budget_s=args.cpu_seconds / 2, rows_per_call=1, bits=bits, k=k, fmt=fmt)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "rows/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": max_ms / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "u32" if esize == 4 else "u16",
            "data": "synthetic",
            "config": workload_config(w, {
                **({} if label == w.name else {"workload": label, "k": k, "format": fmt}),
                "plan": "f32_cluster" if f32_cluster else PLAN_NAME.get(plan, str(plan)),
                "l2": f"inputs rotate over {nbuf} device copies ({nbuf * in_bytes / 1e6:.0f} MB, "
                      f"L2 {l2 / 1e6:.0f} MB)",
                "parallelism": f"replicas x{world} (rows independent, no exchange)"}),
            "us_per_call": avg_launch_s * 1e6,
            "us_per_call_isolated": isolated_s * 1e6 if isolated_s else None,
            "us_per_call_isolated_p10_p50_p90": ([round(float(np.percentile(launch_ms, q)) * 1e3, 2)
                                                  for q in (10, 50, 90)] if launch_ms else None),
            "us_per_call_l2_warm": warm_us,
            "hbm_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": profiled_traffic(kernel, label),
                         "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "launches_timed": args.steps,
                         "duration": ("CUDA events around all timed launches, back to back "
                                      + ("(replayed from a CUDA graph that records the events itself)"
                                         if graph is not None and inner else
                                         "(replayed from a CUDA graph)" if graph is not None else
                                         "(issued from Python)")
                                      + ", / launches"),
                         "ms_per_step_host_events": elapsed_outer_ms / args.steps},
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "cpu_baseline_1core": cpu_1core,
            "per_config": per_config,
            "head": head,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--plan", type=int, default=0,
                    help="TF_TOPK_PLAN_* code: 0 auto, 1 single, 2/4/8/16 cluster, 32 stream, 64 wide")
    ap.add_argument("--dtype", choices=sorted(FORMATS), default="bf16",
                    help="logit format (tf_topk_select for f16 / f32)")
    ap.add_argument("--k", type=int, default=None, help="k (default: the workload's)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="issue the timed launches one by one from Python instead of replaying them as a CUDA graph")
    ap.add_argument("--tables", choices=("all", "head", "none"), default="all",
                    help="after the timed workload: the per-config and draft-head tables, the head table only, or none")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload table (every named workload and sweep points)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
