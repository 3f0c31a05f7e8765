"""Benchmark: GEMM TFLOP/s (2MNK / device time) and % of the GB300 dense tensor peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one GEMM through the C ABI (argument checks, tensor-map encoding, launch, kernel) on
the workload's synthetic inputs, already resident in HBM. W untimed warm-up steps, then exactly K
timed steps; L2 is flushed before every timed step (a 1 GiB device write, 8x the L2, then a
256 MiB device read of the start of that buffer, which writes the flush's dirty lines back to HBM
before the step: the step starts from a cold, clean L2 and is not charged for the flush's
write-back) and each step is timed on its own with CUDA events on the launching stream, so the
flush is outside the timed work. The flush also runs long enough (~200 us) that the host has
enqueued the step's GEMM before the GPU reaches it, so host-side call overhead does not show up as
device time (it does in the end-to-end figure, which copies every step's inputs from pinned host
memory and its result back, pipelined over three streams). Under torchrun each rank runs an independent replica on its own GPU (the GEMM does not
shard across GPUs here: replicas only, no collective), the step time is the max over ranks and
rank 0 prints one JSON line.

--impl reference times the CPU oracle (the plain fp64 definition) on the host cores on a bounded
sample of the same workload per step (a block of output rows), in the same metric and unit.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s (2MNK/device time) and % of GB300 dense tensor peak, 1 GPU"
UNIT = "TFLOP/s"
FLUSH_BYTES = 1 << 30
FLUSH_READ_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "dense_tensor_core_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------------------------------------
# helpers (no GPU needed; the CPU tests exercise them)
# ------------------------------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, world):
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def code_text(src):
    """C/C++ source with its comments removed and whitespace runs collapsed (string and character
    literals kept intact), so that a hash of it changes with the code but not with its comments."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # a literal: copy it whole, escapes included
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# The translation units that launch each benchmarked kernel: with the headers they include they
# define the kernel, and the planner (dtc_gemm.cu) decides its launch.
KERNEL_UNITS = {
    "gemm16_1cta_kernel": ["launch_1cta.cu"],
    "gemm16_2cta_kernel": ["launch_2cta_bf16.cu", "launch_2cta_f16.cu"],
    "gemm16_splitk_kernel": ["launch_splitk.cu"],
    "gemm_mxfp8_kernel": ["launch_mx.cu"],
    "gemm_mxfp8_2cta_kernel": ["launch_mx.cu"],
}


def include_closure(units):
    """The files of `units` and every local header they include, directly or not."""
    seen, todo = set(), list(units)
    while todo:
        f = todo.pop()
        path = os.path.join(CSRC, f)
        if f in seen or not os.path.exists(path):
            continue
        seen.add(f)
        with open(path, encoding="utf-8") as fh:
            todo += re.findall(r'#include\s+"([^"]+)"', fh.read())
    return seen


def source_hash(kernel=None):
    """Hash of the code (comments and layout ignored) of the sources that define `kernel`'s
    launches: its launcher translation units with the headers they include, and the planner's own
    text; of all kernel sources for any other kernel. The DRAM traffic recorded by an ncu capture
    stays valid while that code is unchanged."""
    if kernel in KERNEL_UNITS:
        files = include_closure(KERNEL_UNITS[kernel]) | {"dtc_gemm.cu"}
    else:
        files = {f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))}
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current source of
    that kernel."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(workload, {})
    if e.get("kernel") != kernel or e.get("source_sha") != source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def parse_clocks(csv_text, t0=None, t1=None):
    """Summarise nvidia-smi samples (the recipe's query, with a leading timestamp column)."""
    rows = []
    for line in csv_text.strip().splitlines():
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 10 or not parts[0].replace(".", "", 1).isdigit():
            continue
        try:
            rows.append({"t": float(parts[0]), "sm": float(parts[2].split()[0]),
                         "max": float(parts[3].split()[0]), "hw": parts[6], "hwt": parts[7],
                         "swt": parts[8], "swp": parts[9]})
        except (ValueError, IndexError):
            continue
    window = "timed"
    sel = [r for r in rows if t0 is not None and t0 <= r["t"] <= t1]
    if not sel:
        sel, window = rows, "whole run"
    if not sel:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
    reasons = set()
    for r in sel:
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
            if r[key].lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in sel),
            "sm_max_mhz": max(r["max"] for r in sel), "reasons": sorted(reasons),
            "samples": len(sel), "window": window}


class ClockSampler:
    """nvidia-smi in the background (the recipe's clocks line) with host timestamps."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.out = tempfile.TemporaryFile(mode="w+")

    def __enter__(self):
        cmd = ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
               "--format=csv,noheader", f"-lms", str(self.period)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True, bufsize=1)
        except OSError:
            self.proc = None
        self.lines = []
        if self.proc:
            import threading

            def pump():
                for line in self.proc.stdout:
                    self.lines.append(f"{time.time():.6f}, {line.strip()}")

            self.thread = threading.Thread(target=pump, daemon=True)
            self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(self.period / 1000.0 * 2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def text(self):
        return "\n".join(self.lines)


# NVML clock-event reason bits (nvml.h: nvmlClocksEventReason*), the ones the record names
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def summarise_samples(samples, t0, t1):
    """Clocks record from NVML samples (dicts with t, sm, max, reasons bits): the median SM clock,
    the highest max clock and the active reasons, over the samples taken inside [t0, t1] (the
    timed region), else over all of them."""
    sel = [s for s in samples if t0 <= s["t"] <= t1]
    window = "timed"
    if not sel:
        sel, window = list(samples), "whole run"
    if not sel:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
    bits = 0
    for s in sel:
        bits |= s["reasons"]
    return {"sm_mhz": statistics.median(s["sm"] for s in sel),
            "sm_max_mhz": max(s["max"] for s in sel),
            "reasons": sorted(name for bit, name in NVML_REASONS.items() if bits & bit),
            "samples": len(sel), "window": window,
            "power_w_max": max(s.get("power", 0.0) for s in sel)}


class NvmlSampler:
    """SM clock, power and clock-event reasons of one GPU, read through NVML (the driver's
    libnvidia-ml, loaded with ctypes; reads only) every `period_s` in a background thread, with
    host timestamps. Unavailable (ok() is False) where NVML cannot be loaded."""

    NVML_CLOCK_SM = 1

    def __init__(self, uuid, period_s=0.001):
        self.uuid = uuid
        self.period = period_s
        self.samples = []
        self.lib = None
        self.handle = None
        self._stop = False

    def ok(self):
        return self.handle is not None

    def __enter__(self):
        import ctypes
        import threading

        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return self
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(("GPU-" + str(self.uuid)).encode(), ctypes.byref(h)) != 0:
                lib.nvmlShutdown()
                return self
            self.lib, self.handle = lib, h
        except (OSError, AttributeError):
            return self
        get_reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.NVML_CLOCK_SM, ctypes.byref(mx))

        def poll():
            clk, mw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
            while not self._stop:
                if self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM,
                                                   ctypes.byref(clk)) == 0:
                    self.lib.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(mw))
                    get_reasons(self.handle, ctypes.byref(rs))
                    self.samples.append({"t": time.time(), "sm": float(clk.value),
                                         "max": float(mx.value), "power": mw.value / 1000.0,
                                         "reasons": int(rs.value)})
                time.sleep(self.period)

        self.thread = threading.Thread(target=poll, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        if self.handle is not None:
            time.sleep(2 * self.period)
            self._stop = True
            self.thread.join(timeout=5)
            self.lib.nvmlShutdown()


class Clocks:
    """NVML sampling at 1 ms where available, else nvidia-smi at 20 ms; `record(t0, t1)` gives the
    clocks record of a timed region."""

    def __init__(self, uuid, gpu_index):
        self.nvml = NvmlSampler(uuid)
        self.smi = None
        self.gpu_index = gpu_index

    def __enter__(self):
        self.nvml.__enter__()
        if not self.nvml.ok():
            self.smi = ClockSampler(self.gpu_index).__enter__()
        return self

    def __exit__(self, *exc):
        if self.smi is not None:
            self.smi.__exit__(*exc)
        self.nvml.__exit__(*exc)

    def record(self, t0, t1):
        if self.nvml.ok():
            r = summarise_samples(self.nvml.samples, t0, t1)
            r["source"] = "NVML, 1 ms period"
            return r
        r = parse_clocks(self.smi.text(), t0, t1) if self.smi else parse_clocks("", t0, t1)
        r["source"] = "nvidia-smi, 20 ms period"
        return r


# ------------------------------------------------------------------------------------------------
# CPU oracle leg
# ------------------------------------------------------------------------------------------------

def oracle_rows(w, inputs, rows, cols=None):
    """Run the oracle on the first `rows` output rows (and the first `cols` output columns, all of
    them by default) of workload w; returns seconds taken."""
    import numpy as np

    import oracle

    cols = w.N if cols is None else cols
    t0 = time.perf_counter()
    if w.kind == "mxfp8":
        A, B, sfA, sfB = inputs
        oracle.gemm_bs(A[:rows], B[:cols], sfA[:rows], sfB[:cols], rows, cols, w.K, a_fmt=w.a_fmt,
                       b_fmt=w.b_fmt, block=w.block)
    elif w.kind == "nvfp4":
        A, B, sfA, sfB = inputs
        oracle.gemm_bs(A[:rows], B[:cols], sfA[:rows], sfB[:cols], rows, cols, w.K, a_fmt="e2m1",
                       b_fmt="e2m1", scale="ue4m3", block=16)
    elif w.kind.endswith("_sp24"):
        vals, meta, B = inputs
        Bc = B[:cols] if w.layout[1] == "T" else B[:, :cols]
        oracle.gemm_sp(w.kind[:-5], w.layout, vals[:rows], meta[:rows], np.ascontiguousarray(Bc),
                       rows, cols, w.K)
    else:
        A, B = inputs
        # output rows m are rows of A, or its columns when A is stored [K,M]; output columns n
        # are rows of B when it is stored [N,K], else its columns
        Ar = A[:, :rows] if w.layout[0] == "T" else A[:rows]
        Bc = B[:cols] if w.layout[1] == "T" else B[:, :cols]
        oracle.gemm16(w.kind, w.layout, np.ascontiguousarray(Ar), np.ascontiguousarray(Bc), rows,
                      cols, w.K)
    return time.perf_counter() - t0


def calibrate_rows(w, inputs, target_s):
    """(rows, cols) of C the oracle computes in about target_s seconds.

    Two probes over all N columns separate the fixed cost of a call (decoding B) from the cost per
    output row. When the fixed cost alone would take more than half the budget, the sample keeps
    fewer columns (both costs scale with them), so that many short steps stay short."""
    import oracle

    T = oracle.threads()  # probes are whole multiples of the worker count
    r1, r2 = min(4 * T, w.M), min(16 * T, w.M)
    t1 = oracle_rows(w, inputs, r1)
    t2 = oracle_rows(w, inputs, r2)
    per_row = (t2 - t1) / (r2 - r1) if r2 > r1 else 0.0
    if per_row <= 0.0:
        per_row = t2 / max(r2, 1)
    fixed = max(t1 - r1 * per_row, 0.0)
    cols = w.N
    if fixed > target_s / 2:
        frac = (target_s / 2) / fixed
        cols = max(8, min(w.N, int(w.N * frac)) // 8 * 8)
        per_row *= cols / w.N
        fixed *= cols / w.N
    rows = max(1, min(w.M, int((target_s - fixed) / per_row)))
    return rows, cols


def cpu_baseline(w, inputs, target_s=15.0):
    import oracle

    rows, cols = calibrate_rows(w, inputs, target_s)
    dt = oracle_rows(w, inputs, rows, cols)
    flops = 2.0 * rows * cols * w.K
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{rows} of {w.M} output rows x {cols} of {w.N} columns of {w.name} "
                      f"(full K), {dt:.1f} s"}


# ------------------------------------------------------------------------------------------------
# arms
# ------------------------------------------------------------------------------------------------

def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    inputs = __import__("dense_tensor_core_gb300.workloads", fromlist=["make"]).make(w)
    per_step_budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    rows, cols = calibrate_rows(w, inputs, per_step_budget)
    for _ in range(args.warmup):
        oracle_rows(w, inputs, rows, cols)
    times = [oracle_rows(w, inputs, rows, cols) for _ in range(args.steps)]
    total = sum(times)
    flops = 2.0 * rows * cols * w.K * args.steps
    value = flops / total / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout,
                   "kind": w.kind,
                   "step": f"oracle on {rows} output rows x {cols} columns (bounded sample)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"{rows} of {w.M} output rows x {cols} of {w.N} columns per "
                                   f"step, full K"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def kernel_of(w, plan):
    """The name of the kernel the plan launches (as in the ncu launch list); for the sparse and
    NVFP4 products the GEMM kernel (the step also launches sp24_expand_kernel or
    nvfp4_expand_kernel before it)."""
    if w.kind == "mxfp8":
        return "gemm_mxfp8_2cta_kernel" if plan["variant"] == 2 else "gemm_mxfp8_kernel"
    return {1: "gemm16_1cta_kernel", 2: "gemm16_2cta_kernel",
            3: "gemm16_splitk_kernel"}.get(plan["variant"], str(plan["variant"]))


def run_e2e(w, dtc, host_in, dev_in, C, host_out, step_e2e, stream, steps, dev):
    """Time `steps` pipelined end-to-end steps (H2D inputs, GEMM, D2H result); returns ms."""
    import torch

    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ins = [dev_in, [torch.empty_like(t) for t in dev_in]]
    outs = [C, torch.empty_like(C)]
    hosts = [host_out, torch.empty_like(host_out).pin_memory()]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    gemm_done = [ev(), ev()]  # the GEMM that last read ins[b] / wrote outs[b]
    in_ready = [ev(), ev()]
    out_read = [ev(), ev()]   # the D2H that last read outs[b]
    for e in gemm_done + out_read:
        e.record(stream)

    def one(i):
        b = i % 2
        s_in.wait_event(gemm_done[b])
        with torch.cuda.stream(s_in):
            for h, d in zip(host_in, ins[b]):
                d.copy_(h, non_blocking=True)
        in_ready[b].record(s_in)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_read[b])
        step_e2e(ins[b], outs[b], stream)
        gemm_done[b].record(stream)
        s_out.wait_event(gemm_done[b])
        with torch.cuda.stream(s_out):
            hosts[b].copy_(outs[b], non_blocking=True)
        out_read[b].record(s_out)

    for i in range(2):  # warm the pipeline's buffers and streams
        one(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        one(i)
    s_in.wait_stream(s_out)
    s_in.wait_stream(stream)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1)


def library_context(w, A, B, flush_l2, stream, steps, dev):
    """torch.matmul (cuBLAS) on the same device operands, with the same L2 flush and per-step
    CUDA-event timing: a context figure beside ours, not a baseline and not on our path. None for
    the block-scaled workloads (torch has no product with one E8M0 scale per row per 128 or 32
    K-elements, or one UE4M3 scale per 16, in this row-major scale layout)."""
    import torch

    if w.kind in ("mxfp8", "nvfp4") or w.kind.endswith("_sp24"):
        return None
    a_op = A.t() if w.layout[0] == "T" else A  # A stored [K,M] for TN and TT
    b_op = B.t() if w.layout[1] == "T" else B  # B stored [N,K] for NT and TT
    out = torch.empty((w.M, w.N), dtype=A.dtype, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush_l2(1)
            torch.matmul(a_op, b_op, out=out)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for i in range(steps):
            flush_l2(i)
            starts[i].record(stream)
            torch.matmul(a_op, b_op, out=out)
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.mean(s.elapsed_time(e) for s, e in zip(starts, ends))
    return {"torch_matmul": w.flops / (ms / 1e3) / 1e12, "unit": UNIT, "steps": steps,
            "what": "cuBLAS through torch.matmul on the same device tensors (transposed views "
                    "for the stored layouts), same L2 flush and CUDA-event timing, outside our "
                    "timed region: context only"}


# The benchmark configurations of the pages' workloads (one JSON row each in `configs`), with the
# roofline that bounds each: the tiny and the 1024^3 products are launch- and occupancy-bound, the
# skinny M = 128 product is HBM-bound, the rest tensor-bound.
BENCH_CONFIGS = [
    ("1", "bf16_nt_256x256x512", "latency"),
    ("2", "f16_nn_1024x1024x1024", "latency"),
    ("3", "bf16_nt_4096x4096x8192", "tensor"),
    ("4a", "bf16_nt_8192x8192x8192", "tensor"),
    ("4b", "bf16_nt_128x8192x8192", "hbm"),
    ("5", "mxfp8_nt_4096x4096x8192", "tensor"),
]


def device_inputs(w, dev):
    """The workload's seeded host inputs, on the device: (dev_in, out_dtype, inputs)."""
    import numpy as np
    import torch

    from dense_tensor_core_gb300 import workloads

    inputs = workloads.make(w)
    if w.kind in ("mxfp8", "nvfp4"):
        dev_in = [torch.from_numpy(x).to(dev) for x in inputs]
        return dev_in, torch.bfloat16, inputs
    if w.kind.endswith("_sp24"):  # stored values, metadata, B
        t16 = torch.bfloat16 if w.kind.startswith("bf16") else torch.float16
        vals, meta, B = inputs
        dev_in = [torch.from_numpy(vals.view(np.int16)).view(t16).to(dev),
                  torch.from_numpy(meta).to(dev), torch.from_numpy(B.view(np.int16)).view(t16).to(dev)]
        return dev_in, t16, inputs
    t16 = torch.bfloat16 if w.kind == "bf16" else torch.float16
    dev_in = [torch.from_numpy(x.view(np.int16)).view(t16).to(dev) for x in inputs]
    return dev_in, t16, inputs


def gemm_kwargs(args, w, dtc, dev):
    """Options of the call a user would make for this workload: the automatic plan, and the
    workspace the library asks for (stream-K: zero-filled before first use; block-scaled: the
    repacked scales)."""
    import torch

    if w.kind == "mxfp8":
        kw = dict(a_format=w.a_fmt, b_format=w.b_fmt, scale_block=w.block, variant=args.variant)
        ws_bytes = dtc.gemm_workspace_size("mxfp8", w.M, w.N, w.K, "NT", variant=args.variant,
                                           a_format=w.a_fmt, b_format=w.b_fmt, scale_block=w.block)
        if ws_bytes:
            kw["workspace"] = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        return kw
    base = w.kind[:-5] if w.kind.endswith("_sp24") else "bf16" if w.kind == "nvfp4" else w.kind
    kw = dict(layout=w.layout, variant=args.variant, split_k=args.split_k, tile_n=args.tile_n)
    if args.stream_k != 2:
        ws_bytes = dtc.gemm_workspace_size(base, w.M, w.N, w.K, w.layout, variant=args.variant,
                                           tile_n=args.tile_n, stream_k=args.stream_k)
        if ws_bytes:
            kw.update(workspace=torch.zeros(ws_bytes, dtype=torch.uint8, device=dev),
                      stream_k=args.stream_k)
    if w.kind.endswith("_sp24"):  # the expanded A, and the dense product's stream-K workspace
        kw["sk_workspace"] = kw.pop("workspace", None)
        kw["sp_workspace"] = torch.empty(dtc.gemm_sp_workspace_size(base, w.M, w.K),
                                         dtype=torch.uint8, device=dev)
    if w.kind == "nvfp4":  # the operands expanded to bf16, and the product's stream-K workspace
        kw.pop("layout")
        kw["sk_workspace"] = kw.pop("workspace", None)
        kw["nv_workspace"] = torch.empty(dtc.gemm_nvfp4_workspace_size(w.M, w.N, w.K),
                                         dtype=torch.uint8, device=dev)
    return kw


def call(dtc, w, ins, C, kw, stream):
    if w.kind == "mxfp8":
        dtc.gemm_ex("mxfp8", ins[0], ins[1], C, sfA=ins[2], sfB=ins[3], stream=stream, **kw)
    elif w.kind.endswith("_sp24"):
        kw = dict(kw)
        dtc.gemm_sp(w.kind[:-5], ins[0], ins[1], ins[2], C, workspace=kw.pop("sp_workspace"),
                    stream=stream, **kw)
    elif w.kind == "nvfp4":
        kw = dict(kw)
        dtc.gemm_nvfp4(ins[0], ins[1], ins[2], ins[3], C, workspace=kw.pop("nv_workspace"),
                       stream=stream, **kw)
    else:
        dtc.gemm_ex(w.kind, ins[0], ins[1], C, stream=stream, **kw)


def plan_of(dtc, w, kw):
    keys = ("layout", "variant", "split_k", "tile_n", "workspace", "stream_k", "a_format",
            "b_format", "scale_block")
    kw = dict(kw)
    if w.kind.endswith("_sp24") or w.kind == "nvfp4":  # the dense product on the expanded operands
        kw["workspace"] = kw.pop("sk_workspace", None)
        base = "bf16" if w.kind == "nvfp4" else w.kind[:-5]
        return dtc.gemm_plan(base, w.M, w.N, w.K, **{k: v for k, v in kw.items() if k in keys})
    return dtc.gemm_plan(w.kind, w.M, w.N, w.K, **{k: v for k, v in kw.items() if k in keys})


def launches_per_step(w, plan):
    """Our kernels in one step: the GEMM, plus the 2:4 or NVFP4 expansion or the scale
    repacking."""
    return 2 if w.kind.endswith("_sp24") or w.kind == "nvfp4" or plan.get("sf_packed") else 1


def timed_steps(step, flush_l2, steps, warmup, stream, dev, world):
    """W warm-up steps, then `steps` timed ones, each bracketed by CUDA events on the launching
    stream after an L2 flush outside the events; returns (per-step ms, t0, t1 host times)."""
    import torch

    for _ in range(warmup):
        flush_l2(1)
        step()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(steps):
        flush_l2(i)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t1 = time.time()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], t0, t1


def roofline_of(w, kernel_ms, bound, kernel_name, peaks, peak_src):
    """The roofline record of one launch of `kernel_name` on workload w."""
    if bound == "hbm":
        bw = w.min_bytes / (kernel_ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": bw, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": bw / peaks["hbm_gbs"], "traffic": recorded_traffic(w.name, kernel_name),
                "kernel": kernel_name, "peak_source": f"{peak_src} HBM copy bandwidth",
                "algorithmic_bytes_per_launch": w.min_bytes}
    achieved = w.flops / (kernel_ms / 1e3) / 1e12
    if w.kind == "mxfp8":
        # fp8 dense rate = 2x the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s)
        peak = 2.0 * peaks["bf16_tflops"]
        note = f"2 x {peak_src} bf16 burst (nominal fp8:bf16 ratio)"
    elif w.kind == "nvfp4":
        peak = peaks["bf16_tflops"]
        note = (f"{peak_src} bf16 burst: the NVFP4 product runs on the bf16 tensor cores after "
                "the exact expansion of its operands (the fp4-rate kind is not used)")
    else:
        peak = peaks["bf16_tflops"]
        note = f"{peak_src} bf16 burst (kernel timed alone)"
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "traffic": recorded_traffic(w.name, kernel_name),
            "kernel": kernel_name, "peak_source": note, "algorithmic_flops_per_launch": w.flops}


def run_ours(args, w):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from dense_tensor_core_gb300 import build as cuda_build

    cuda_build.build()
    import dense_tensor_core_gb300 as dtc
    from dense_tensor_core_gb300 import workloads

    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_read = flush[: FLUSH_READ_BYTES // 4]
    flush_sink = torch.zeros((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(i):
        flush.fill_(float(i))
        torch.sum(flush_read, dim=0, out=flush_sink)  # evicts (writes back) the dirty lines

    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()
    launches = 0
    with Clocks(getattr(props, "uuid", ""), local if world > 1 else 0) as clk:
        dev_in, out_dtype, inputs = device_inputs(w, dev)
        C = torch.empty((w.M, w.N), dtype=out_dtype, device=dev)
        kw = gemm_kwargs(args, w, dtc, dev)
        plan = plan_of(dtc, w, kw)
        step_ms, t0, t1 = timed_steps(lambda: call(dtc, w, dev_in, C, kw, stream), flush_l2,
                                      args.steps, args.warmup, stream, dev, world)
        launches += args.steps * launches_per_step(w, plan)
        dtc.gemm_stream_status(stream)
        clocks = clk.record(t0, t1)

        total_ms = max_over_ranks(sum(step_ms), world)
        ms_per_step = total_ms / args.steps
        value = world * float(w.flops) * args.steps / (total_ms / 1e3) / 1e12
        kernel_ms = statistics.mean(step_ms)  # one launch of our kernel per step
        kernel_name = kernel_of(w, plan)

        # End to end through the public call with host buffers: every step copies its inputs
        # from pinned host memory (H2D), runs the GEMM and copies the result back (D2H). The steps
        # are pipelined as a streaming user would run them: two device copies of the inputs and
        # of C, H2D on one stream, the GEMM on another, D2H on a third, so step i+1's inputs cross
        # the host link while step i computes and step i-1's result comes back. Events order
        # every reuse of a buffer after its previous reader.
        host_in = [t.cpu().pin_memory() for t in dev_in]
        host_out = torch.empty((w.M, w.N), dtype=out_dtype).pin_memory()
        e2e_steps = max(1, min(args.steps, 20))  # each step moves the workload over the host link
        e2e_ms = run_e2e(w, dtc, host_in, dev_in, C, host_out,
                         lambda ins, Cout, st: call(dtc, w, ins, Cout, kw, st), stream, e2e_steps,
                         dev)
        launches += e2e_steps * launches_per_step(w, plan)
        e2e_ms = max_over_ranks(e2e_ms, world)
        dtc.gemm_stream_status(stream)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = host_out.numel() * host_out.element_size()
        e2e_value = world * float(w.flops) * e2e_steps / (e2e_ms / 1e3) / 1e12
        library = library_context(w, dev_in[0], dev_in[1], flush_l2, stream,
                                  min(args.steps, 50), dev)
        del host_in, host_out

        # every benchmark configuration of the pages' workloads, timed the same way
        configs = {}
        if not args.no_configs and world == 1:
            cfg_steps = max(20, min(args.steps, 200))
            for cid, name, bound in BENCH_CONFIGS:
                cw = workloads.WORKLOADS[name]
                if name == w.name:
                    cms, cplan, ct0, ct1, cname, clib = kernel_ms, plan, t0, t1, kernel_name, library
                    csteps = args.steps
                else:
                    cin, cdt, _ = device_inputs(cw, dev)
                    cC = torch.empty((cw.M, cw.N), dtype=cdt, device=dev)
                    ckw = gemm_kwargs(args, cw, dtc, dev)
                    cplan = plan_of(dtc, cw, ckw)
                    cms_list, ct0, ct1 = timed_steps(
                        lambda: call(dtc, cw, cin, cC, ckw, stream), flush_l2, cfg_steps, 5,
                        stream, dev, world)
                    launches += cfg_steps * launches_per_step(cw, cplan)
                    dtc.gemm_stream_status(stream)
                    cms = statistics.mean(cms_list)
                    cname = kernel_of(cw, cplan)
                    clib = library_context(cw, cin[0], cin[1], flush_l2, stream, cfg_steps, dev)
                    csteps = cfg_steps
                    del cin, cC, ckw
                rl = roofline_of(cw, cms, "hbm" if bound == "hbm" else "tensor", cname, peaks,
                                 peak_src)
                configs[cid] = {
                    "workload": name, "bound": bound, "kernel": cname, "steps": csteps,
                    "us_per_launch": 1e3 * cms, "tflops": cw.flops / (cms / 1e3) / 1e12,
                    "gbs_compulsory": cw.min_bytes / (cms / 1e3) / 1e9,
                    "frac": rl["frac"], "frac_of": f'{rl["peak"]:.1f} {rl["unit"]} ({rl["peak_source"]})',
                    "tile": f"{cplan['tile_m']}x{cplan['tile_n']}x{cplan['tile_k']}",
                    "split_k": cplan["split_k"], "stream_k_tiles": cplan["sk_tiles"],
                    "library_context_tflops": clib["torch_matmul"] if clib else None,
                    "clocks": clk.record(ct0, ct1),
                }

    if rank != 0:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return 0

    bound = "hbm" if (w.name == "bf16_nt_128x8192x8192" or (w.M <= 256 and w.kind != "mxfp8")) \
        else "tensor"
    roofline = roofline_of(w, kernel_ms, bound, kernel_name, peaks, peak_src)
    achieved_tflops = w.flops / (kernel_ms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": (w.kind[:-5] if w.kind.endswith("_sp24") else "bf16" if w.kind in ("bf16", "nvfp4")
                  else "f16" if w.kind == "f16"
                  else w.a_fmt if w.a_fmt == w.b_fmt else f"{w.a_fmt}x{w.b_fmt}"),
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "layout": w.layout,
                   "kind": w.kind, "variant": kernel_name,
                   **({"scale_block": w.block} if w.kind == "mxfp8" else {}),
                   **({"inputs": "e2m1 x e2m1, UE4M3 scales per 16, expanded to bf16"}
                      if w.kind == "nvfp4" else {}),
                   "tile": f"{plan['tile_m']}x{plan['tile_n']}x{plan['tile_k']}",
                   "stages": plan["stages"], "split_k": plan["split_k"], "ctas": plan["ctas"],
                   "stream_k_tiles": plan["sk_tiles"],
                   "cluster": plan["cluster"],
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed before every timed step, outside the step's CUDA-event "
                         "pair: 1 GiB device write, then a 256 MiB device read that writes the "
                         "flush's dirty lines back (cold, clean L2)",
                   "pct_of_dense_peak_nominal": 100.0 * achieved_tflops /
                   (4500.0 if w.kind == "mxfp8" else 2250.0),
                   "timed_wall_ms": 1e3 * (t1 - t0)},
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "mode": "pipelined: step i+1's H2D and step i-1's D2H overlap step i's GEMM "
                        "(3 streams, 2 device buffers); pinned host memory"},
        # our kernels per timed step of the headline: the GEMM (and the sparse expansion or the
        # scale repacking)
        "gpu_launches": args.steps * launches_per_step(w, plan),
        "gpu_launches_whole_run": launches,  # with the end-to-end steps and the other configs
        "clocks": clocks,
        "library_context": library,
    }
    if configs:
        line["configs"] = configs
    if not args.skip_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inputs, target_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None, help="workload name (default: the headline)")
    p.add_argument("--variant", type=int, default=0, help="0 auto, 1 one-CTA, 2 CTA pair, 3 split-K")
    p.add_argument("--split-k", type=int, default=0)
    p.add_argument("--tile-n", type=int, default=0, help="force the N-tile (256 or 224)")
    p.add_argument("--stream-k", type=int, default=0, choices=[0, 1, 2],
                   help="stream-K on CTA pairs: 0 auto (a workspace is passed when it helps), "
                        "1 required, 2 off")
    p.add_argument("--no-configs", action="store_true",
                   help="time only the chosen workload (not every benchmark configuration)")
    p.add_argument("--skip-cpu-baseline", action="store_true",
                   help="omit the oracle timing (profiling runs)")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    from dense_tensor_core_gb300 import workloads

    w = workloads.WORKLOADS[args.workload or workloads.HEADLINE]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
