"""Benchmark of the blockwise-FP8 linear training hot path on GB300.

One step = one Float8BlockwiseLinear forward+backward on the dense workload
(M=16384 tokens, K=5120, N=8192): 1x128 quantization of x, 128x128
quantization of W, y = x W^T, 1x128 quantization of dy, dx = dy W, colwise
1x128 quantization of dy and x, dW = dy^T x -- eight library launches.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is the step's GEMM work (3 x 2MNK flops) over
the device time of whole steps (quantizers included), summed over ranks.
Inputs (520 MB bf16) and the step's outputs exceed the 129 MB L2, so no flush
is needed between steps.  Roofline fractions are against the burst fp8 peak
(the measured burst bf16 GEMM rate x 2; the timed regions are tens of
milliseconds at full clock), with the sustained figure beside it.  Further
sections of the same line time the two large-token workloads (M = 128000),
the toy FFN step, the MXFP8 MoE step and the MXFP8 dense linear.
`--impl reference` times the CPU oracle on a bounded sample of the dense
workload instead.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "blockwise-FP8 GEMM TFLOPS (fwd+dgrad+wgrad) & quant GB/s, % of GB300 roofline"
M, K, N = 16384, 5120, 8192
WORKLOAD = f"dense Float8BlockwiseLinear fwd+bwd, M={M} K={K} N={N}, x~N(0,1) W~N(0,0.02) dy~N(0,1e-3), seed 2"

# Fallback peaks (used only when MEASURED_PEAKS.json is absent).
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
FP8_OVER_BF16 = 2.0  # nominal dense ratio 4.5 / 2.25 PFLOP/s


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sustained": p["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16": FALLBACK_BF16_TFLOPS, "bf16_sustained": FALLBACK_BF16_TFLOPS_SUSTAINED,
            "source": "fallback"}


# ---------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """SM clock and clock-event reasons sampled on a thread while the timed
    region runs: through NVML (ctypes, every ~2 ms, so a
    region of tens of milliseconds still gets many samples), or through
    `nvidia-smi -lms 50` where NVML cannot be loaded.  Reads only; changes no
    setting of the GPU."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int, uuid: str | None = None, period_s: float = 0.002):
        self.gpu, self.uuid, self.period = gpu_index, uuid, period_s
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.nvml = None
        self.proc = None
        self.path = os.path.join("/tmp", f"fp8bw_clocks_{os.getpid()}.csv")

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + self.uuid).encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.gpu, ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return lib, h, reasons_fn

    def _loop(self):
        import ctypes
        lib, h, reasons_fn = self.nvml
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(float(clk.value))
            if reasons_fn(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            self.stop.wait(self.period)

    def __enter__(self):
        import threading
        try:
            self.nvml = self._nvml_open()
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
        except (OSError, AttributeError):
            self.nvml = None
            try:
                self.f = open(self.path, "w")
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={CLOCK_FIELDS}",
                                              "--format=csv,noheader,nounits", "-lms", "50"],
                                             stdout=self.f, stderr=subprocess.DEVNULL)
            except OSError:
                self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            try:
                self.nvml[0].nvmlShutdown()
            except OSError:
                pass
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.nvml is None and self.proc is not None and os.path.exists(self.path):
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        self.samples.append(float(parts[1]))
                        self.max_mhz = float(parts[2])
                    except ValueError:
                        continue
                    for name, val in zip(names, parts[5:9]):
                        if val.lower().startswith("active"):
                            self.reasons.add(name)
            os.unlink(self.path)
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml" if self.nvml is not None else "nvidia-smi"}


# ---------------------------------------------------------------- distributed plumbing

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("FP8BW_BENCH_GLOO") is None else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)

_DENSE = None


def dense_inputs():
    global _DENSE
    if _DENSE is None:
        from mxfp8_precision_gemms_fp8bw_gb300 import inputs
        _DENSE = inputs.dense()
    return _DENSE


def oracle_sample(rows: int, w_rows: int):
    """The oracle on a bounded sample of the dense workload: the first `rows`
    tokens of x and dy and the first `w_rows` output features of W -- every
    quantization of the step on that sample (rowwise and colwise for x and dy,
    128x128 for W) and the three GEMMs restricted to it (dgrad and wgrad
    contract over the sampled features / tokens only).
    Returns (seconds, gemm flops, threads, quantizer seconds, quantizer
    algorithmic bytes): the five quantizations are also timed on their own,
    since quantizers are reported in GB/s apart from the GEMMs."""
    import oracle
    from mxfp8_precision_gemms_fp8bw_gb300 import inputs

    t = dense_inputs()
    x = inputs.bf16_to_f32_numpy(t.x[:rows])
    w = inputs.bf16_to_f32_numpy(t.w[:w_rows])
    dy = inputs.bf16_to_f32_numpy(t.dy[:rows, :w_rows])
    qsecs = 0.0

    def quant(fn, a):
        nonlocal qsecs
        q0 = time.perf_counter()
        out = fn(a)
        qsecs += time.perf_counter() - q0
        return out

    t0 = time.perf_counter()
    xq, xs = quant(oracle.quant_1x128_row, x)
    wq, _, ws = quant(oracle.quant_128x128, w)
    y = oracle.gemm_fwd(xq, xs, wq, ws)
    dyq, dys = quant(oracle.quant_1x128_row, dy)
    dx = oracle.gemm_dgrad(dyq, dys, wq, ws)
    dyqT, dysT = quant(oracle.quant_1x128_col, dy)
    xqT, xsT = quant(oracle.quant_1x128_col, x)
    dW = oracle.gemm_wgrad(dyqT, dysT, xqT, xsT)
    secs = time.perf_counter() - t0
    # Algorithmic bytes of the five calls: bf16 read, e4m3 written, fp32
    # scales (one per 128 elements for 1x128, one per 128x128 tile for W).
    qbytes = 2 * (rows * K + rows * w_rows) * (3 + 4 / 128) + w_rows * K * (3 + 4 / (128 * 128))
    assert y.shape == (rows, w_rows) and dx.shape == (rows, K) and dW.shape == (w_rows, K)
    threads = os.cpu_count() or 1
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            threads = max(i.get("num_threads", 1) for i in info)
    except ImportError:
        pass
    return secs, 6 * rows * w_rows * K, threads, qsecs, qbytes


def sample_desc(rows, w_rows):
    return (f"first {rows} of {M} tokens and first {w_rows} of {N} output features: all five quantizations "
            f"and the three GEMMs on that sample (float64 numpy oracle), GEMM flops / wall time")


REF_SAMPLE = (128, 1024)      # per step of --impl reference (a second or two), shrunk for long runs
REF_BUDGET_S = 150.0          # wall-time target of a whole --impl reference run
CPU_SAMPLE = (2048, 8192)  # cpu_baseline of the GPU arm (about ten seconds of CPU work on 16 cores)


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    rows, w_rows = REF_SAMPLE
    # The sampled output features are halved (down to one 128-block) until
    # all warm-up and timed steps fit in about REF_BUDGET_S seconds at a
    # conservative per-step estimate.  The metric is flops per second, so the
    # sample size changes the work per step, not the unit.
    est = lambda w: 2.5 * w / 1024 + 0.1  # noqa: E731  (seconds per step, 8 host cores)
    while w_rows > 128 and est(w_rows) * (args.steps + args.warmup) > REF_BUDGET_S:
        w_rows //= 2
    vals = []
    for _ in range(args.warmup):
        oracle_sample(rows, w_rows)
    secs_all = []
    for _ in range(args.steps):
        secs, flops, threads, _, _ = oracle_sample(rows, w_rows)
        secs_all.append(secs)
        vals.append(flops / secs / 1e12)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(secs_all) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample_desc(rows, w_rows)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- GPU arm

def run_ours(args, world, rank, local):
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
    from mxfp8_precision_gemms_fp8bw_gb300.linear import BlockwiseLinearWorkspace

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.lib(build_if_missing=True)
    peaks = load_peaks()

    t = dense_inputs()
    x_h, w_h, dy_h = t.x.pin_memory(), t.w.pin_memory(), t.dy.pin_memory()
    x, w, dy = x_h.to(dev), w_h.to(dev), dy_h.to(dev)
    ws = BlockwiseLinearWorkspace(M, N, K, device=dev)
    stream = torch.cuda.current_stream(dev)
    kern = ws.kernels(x, w, dy)
    names = [n for n, _ in kern]
    algo = ws.algorithmic()

    for _ in range(args.warmup):
        ws.step(x, w, dy)
    B.fp8bw_sync_status()

    # Timed region: K whole steps, with an event between consecutive launches.
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local, device_uuid(dev)) as clk:
        ms_step, per_kernel = time_kernels(kern, args.steps, stream)
    barrier(world)
    B.fp8bw_sync_status()
    ms_step = max_over_ranks(world, ms_step, dev)

    gemm_flops = 3 * 2 * M * N * K
    value = gemm_flops * world / (ms_step * 1e-3) / 1e12

    # The timed region lasts tens of milliseconds at full clock, so the burst
    # figure is the denominator; the sustained one is reported beside it.
    fp8_peak = peaks["bf16"] * FP8_OVER_BF16
    fp8_sustained = peaks["bf16_sustained"] * FP8_OVER_BF16
    kernels = kernel_table(per_kernel, algo, fp8_peak, peaks["hbm_gbs"])
    gemm_ms = sum(per_kernel[n] for n in names if algo[n][0] == "flops")
    quant_ms = sum(per_kernel[n] for n in names if algo[n][0] == "bytes")
    quant_bytes = sum(algo[n][1] for n in names if algo[n][0] == "bytes")

    dom = max((n for n in names if algo[n][0] == "flops"), key=lambda n: per_kernel[n])
    dom_ach = algo[dom][1] / (per_kernel[dom] * 1e-3) / 1e12
    traffic = load_traffic(dom)
    roofline = {"kernel": dom, "bound": "tensor", "achieved": round(dom_ach, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(dom_ach / fp8_peak, 4), "traffic": traffic,
                "peak_source": f"{peaks['source']} burst bf16 x {FP8_OVER_BF16:g} (nominal fp8/bf16 ratio)",
                "peak_sustained": round(fp8_sustained, 1), "frac_vs_sustained": round(dom_ach / fp8_sustained, 4)}

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned memory, runs, and copies y, dx, dW back, with the
    # copies of neighbouring steps overlapping the kernels (PipelinedLinearSteps).
    from mxfp8_precision_gemms_fp8bw_gb300.linear import PipelinedLinearSteps
    y_h = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    dx_h = torch.empty((M, K), dtype=torch.bfloat16, pin_memory=True)
    dW_h = torch.empty((N, K), dtype=torch.bfloat16, pin_memory=True)
    pipe = PipelinedLinearSteps(M, N, K, device=dev)
    e2e_steps = max(1, min(args.steps, 20))
    for _ in range(2):
        pipe.step(x_h, w_h, dy_h, y_h, dx_h, dW_h)
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    barrier(world)
    # the first upload starts after e0 (upload stream); the last download ends before e1
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.up)
    for _ in range(e2e_steps):
        pipe.step(x_h, w_h, dy_h, y_h, dx_h, dW_h)
    pipe.down.wait_stream(pipe.comp)
    e1.record(pipe.down)
    pipe.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1) / e2e_steps, dev)
    del pipe
    h2d = (x.numel() + w.numel() + dy.numel()) * 2
    d2h = (y_h.numel() + dx_h.numel() + dW_h.numel()) * 2

    sec_steps = max(10, args.steps // 3)
    large = [run_large_token(dev, i, sec_steps, args.warmup, fp8_peak, peaks["hbm_gbs"], world) for i in (0, 1)]
    ffn = run_ffn(dev, sec_steps, args.warmup, fp8_peak, peaks["hbm_gbs"], world)
    chain = run_chain_epilogue_quant(dev, sec_steps, args.warmup, fp8_peak, peaks["hbm_gbs"], world)
    moe = None if args.no_moe else run_moe(dev, max(10, args.steps // 3), args.warmup, fp8_peak, peaks["hbm_gbs"],
                                           world)
    mx_dense = None if args.no_moe else run_moe(dev, max(10, args.steps // 3), args.warmup, fp8_peak,
                                                peaks["hbm_gbs"], world, dense=True)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows, w_rows = CPU_SAMPLE
        secs, flops, threads, qsecs, qbytes = oracle_sample(rows, w_rows)
        cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": sample_desc(rows, w_rows), "seconds": round(secs, 2),
               "gemm_tflops": round(flops / (secs - qsecs) / 1e12, 4),
               "quant_gbs": round(qbytes / qsecs / 1e9, 3)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp8_e4m3 (fp32 accumulate, bf16 out)", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "parallelism": f"replicas x{world}",
                       "l2": "inputs 520 MB and outputs exceed the 129 MB L2; no flush"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(gemm_flops * world / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": len(kern) * args.steps,
            "clocks": clk.summary(),
            "gemm_tflops": round(gemm_flops / (gemm_ms * 1e-3) / 1e12, 1),
            "quant_gbs": round(quant_bytes / (quant_ms * 1e-3) / 1e9, 1),
            "hbm_peak_gbs": peaks["hbm_gbs"],
            "kernels": kernels,
            "linear_us": linear_us(per_kernel, ["quant_1x128_rowcol(x)", "quant_128x128(W)", "gemm_fwd"]),
            "large_token": large,
            "toy_ffn": ffn,
            "linear_chain_epilogue_quant": chain,
            "mxfp8_moe": moe,
            "mxfp8_dense": mx_dense,
        }
        print(json.dumps(line))
    return 0


def device_uuid(dev):
    try:
        import torch
        return str(torch.cuda.get_device_properties(dev).uuid)
    except (AttributeError, RuntimeError):
        return None


def linear_us(per_kernel, fwd_names):
    """Per-linear end-to-end times in the microbenchmark columns of PR #3037:
    forward (its quantizations and GEMM) and forward + backward (the whole
    step), in microseconds, from the per-launch event times."""
    return {"fwd_us": round(1e3 * sum(per_kernel[n] for n in fwd_names), 1),
            "fwd_bwd_us": round(1e3 * sum(per_kernel.values()), 1)}


def time_kernels(kern, steps, stream):
    """Times `steps` passes over the (name, fn) list with an event between
    consecutive launches; returns (ms per pass, {name: mean ms})."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kern) + 1)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(steps):
        evs[s][0].record(stream)
        for i, (_, fn) in enumerate(kern):
            fn()
            evs[s][i + 1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    per = {n: statistics.mean(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps))
           for i, (n, _) in enumerate(kern)}
    return start.elapsed_time(end) / steps, per


def kernel_table(per, algo, fp8_peak, hbm_peak):
    out = {}
    for n, ms in per.items():
        kind, amount = algo[n]
        if kind is None:
            out[n] = {"ms": round(ms, 4), "note": "model torch op, not a library call"}
        elif kind == "flops":
            ach = amount / (ms * 1e-3) / 1e12
            out[n] = {"ms": round(ms, 4), "TFLOP/s": round(ach, 1), "frac": round(ach / fp8_peak, 3)}
        else:
            ach = amount / (ms * 1e-3) / 1e9
            out[n] = {"ms": round(ms, 4), "GB/s": round(ach, 1), "frac": round(ach / hbm_peak, 3)}
    return out


def run_moe(dev, steps, warmup, fp8_peak, hbm_peak, world, dense: bool = False):
    """The MXFP8 MoE grouped linear step (M=16384 tokens over 8 experts,
    K=5120, N=8192): six library calls (three fused row + column MX
    quantizations and three grouped GEMMs), timed like the dense step.  With
    dense=True, the MXFP8 dense linear instead: the same six calls with one
    group on the dense workload's x, W, dy (M=16384, K=5120, N=8192)."""
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
    from mxfp8_precision_gemms_fp8bw_gb300 import inputs
    from mxfp8_precision_gemms_fp8bw_gb300.linear import MxMoEWorkspace

    if dense:
        t = dense_inputs()
        M, K = t.x.shape
        N = t.w.shape[0]
        t = inputs.MoEInputs(x=t.x, w=t.w.reshape(1, N, K), dy=t.dy, group_end=np.array([M], np.int32))
    else:
        t = inputs.moe()
    G, N, K = t.w.shape
    M = t.x.shape[0]
    x, w, dy = t.x.to(dev), t.w.to(dev), t.dy.to(dev)
    ge = torch.from_numpy(t.group_end).to(dev)
    ws = MxMoEWorkspace(M, N, K, G, device=dev)
    kern = ws.kernels(x, w, dy, ge)
    for _ in range(warmup):
        ws.step(x, w, dy, ge)
    B.fp8bw_sync_status()
    barrier(world)
    ms_step, per = time_kernels(kern, steps, torch.cuda.current_stream(dev))
    B.fp8bw_sync_status()
    ms_step = max_over_ranks(world, ms_step, dev)
    algo = ws.algorithmic()
    flops = 3 * 2 * M * N * K
    gemm_names = [n for n in per if algo[n][0] == "flops"]
    dom = max(gemm_names, key=lambda n: per[n])
    dom_ach = algo[dom][1] / (per[dom] * 1e-3) / 1e12
    sizes = [int(v) for v in np.diff(np.concatenate([[0], t.group_end]))]
    workload = (f"MXFP8 dense linear fwd+bwd (one group), M={M} K={K} N={N}, the dense workload's x W dy, "
                f"1x32 E8M0 RCEIL, seed 2" if dense else
                f"MXFP8 MoE grouped linear fwd+bwd, M={M} tokens over G={G} experts (sizes {sizes}), "
                f"K={K}, N={N}, 1x32 E8M0 RCEIL, seed 4")
    return {
        "workload": workload,
        "value": round(flops * world / (ms_step * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_step": round(ms_step, 4), "steps": steps, "gpu_launches": len(kern) * steps,
        "gemm_tflops": round(flops / (sum(per[n] for n in gemm_names) * 1e-3) / 1e12, 1),
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(dom_ach, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(dom_ach / fp8_peak, 4),
                     "traffic": load_traffic(("mxfp8_dense/" if dense else "") + dom)},
        "kernels": kernel_table(per, algo, fp8_peak, hbm_peak),
        "linear_us": linear_us(per, ["mx_quant_1x32_rowcol(x)", "mx_quant_1x32_rowcol(W)", "mx_grouped_fwd"]),
    }


def section_from_times(workload, per, algo, flops, ms_step, steps, fp8_peak, hbm_peak, fwd_names, world, extra=None,
                       traffic_key=None):
    """One bench section: whole-step TFLOP/s, per-call times and roofline
    fractions, the dominant GEMM, and the per-linear microseconds.  The
    dominant GEMM's DRAM traffic comes from the ncu summary under
    `traffic_key` (``<section>/<kernel>``) when one was taken on this shape."""
    gemm_names = [n for n in per if algo[n][0] == "flops"]
    dom = max(gemm_names, key=lambda n: per[n])
    dom_ach = algo[dom][1] / (per[dom] * 1e-3) / 1e12
    sec = {
        "workload": workload,
        "value": round(flops * world / (ms_step * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_step": round(ms_step, 4), "steps": steps,
        "gpu_launches": sum(1 for n in per if algo[n][0] is not None) * steps,
        "gemm_tflops": round(flops / (sum(per[n] for n in gemm_names) * 1e-3) / 1e12, 1),
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(dom_ach, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(dom_ach / fp8_peak, 4),
                     "traffic": load_traffic(f"{traffic_key}/{dom}") if traffic_key else None},
        "kernels": kernel_table(per, algo, fp8_peak, hbm_peak),
        "linear_us": linear_us(per, fwd_names),
    }
    if extra:
        sec.update(extra)
    return sec


def run_large_token(dev, which, steps, warmup, fp8_peak, hbm_peak, world):
    """The blockwise linear on a large-token workload (M = 128000 tokens, so
    wgrad contracts over 128000): the six-call step of the dense workload.
    Inputs are seeded normals with the workload's distributions drawn on the
    device (the parity tests use the host-drawn seeded inputs)."""
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
    from mxfp8_precision_gemms_fp8bw_gb300 import inputs
    from mxfp8_precision_gemms_fp8bw_gb300.linear import BlockwiseLinearWorkspace

    Mt, Kt, Nt = inputs.LARGE_SHAPES[which]
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    draw = lambda shape, std: (torch.randn(shape, generator=g, device=dev) * std).bfloat16()  # noqa: E731
    x, w, dy = draw((Mt, Kt), 1.0), draw((Nt, Kt), 0.02), draw((Mt, Nt), 1e-3)
    ws = BlockwiseLinearWorkspace(Mt, Nt, Kt, device=dev)
    kern = ws.kernels(x, w, dy)
    for _ in range(warmup):
        ws.step(x, w, dy)
    B.fp8bw_sync_status()
    barrier(world)
    ms_step, per = time_kernels(kern, steps, torch.cuda.current_stream(dev))
    B.fp8bw_sync_status()
    ms_step = max_over_ranks(world, ms_step, dev)
    workload = (f"large-token dense Float8BlockwiseLinear fwd+bwd, M={Mt} K={Kt} N={Nt} (wgrad contracts over "
                f"{Mt} tokens), x~N(0,1) W~N(0,0.02) dy~N(0,1e-3) drawn on the device, seed 3")
    sec = section_from_times(workload, per, ws.algorithmic(), 6 * Mt * Nt * Kt, ms_step, steps, fp8_peak, hbm_peak,
                             ["quant_1x128_rowcol(x)", "quant_128x128(W)", "gemm_fwd"], world,
                             traffic_key=f"large{which}")
    del x, w, dy, ws, kern
    torch.cuda.empty_cache()
    return sec


def run_ffn(dev, steps, warmup, fp8_peak, hbm_peak, world):
    """The toy FFN of PR #4295 (out = out_proj(silu(w1 x) * (w2 x)), tokens
    4096, dim 2048, hidden 8192, 1 % outlier rows in x): one forward+backward
    step of nine blockwise GEMMs, their quantizations and the model's own
    elementwise activation (torch ops, timed as part of the step)."""
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
    from mxfp8_precision_gemms_fp8bw_gb300 import inputs
    from mxfp8_precision_gemms_fp8bw_gb300.linear import ToyFFNStep

    t = inputs.ffn()
    M_, D_ = t.x.shape
    H_ = t.w1.shape[0]
    x, w1, w2, wo, dy = (a.to(dev) for a in (t.x, t.w1, t.w2, t.out_proj, t.dy))
    ws = ToyFFNStep(M_, D_, H_, device=dev)
    kern = ws.kernels(x, w1, w2, wo, dy)
    for _ in range(warmup):
        ws.step(x, w1, w2, wo, dy)
    B.fp8bw_sync_status()
    barrier(world)
    ms_step, per = time_kernels(kern, steps, torch.cuda.current_stream(dev))
    B.fp8bw_sync_status()
    ms_step = max_over_ranks(world, ms_step, dev)
    algo = ws.algorithmic()
    flops = sum(v for k, v in algo.values() if k == "flops")
    workload = (f"toy FFN out_proj(silu(w1 x) * (w2 x)) fwd+bwd, tokens={M_} dim={D_} hidden={H_}, x~N(0,1) with "
                f"{len(t.outlier_rows)} outlier rows x10^U(1,2), weights~N(0,0.02), dy~N(0,1e-3), seed 1")
    torch_ms = sum(v for n, v in per.items() if algo[n][0] is None)
    return section_from_times(workload, per, algo, flops, ms_step, steps, fp8_peak, hbm_peak,
                              ["quant_1x128_rowcol(x)", "quant_128x128(w1)", "quant_128x128(w2)", "gemm_fwd(w1)",
                               "gemm_fwd(w2)", "act silu*mul (torch)", "quant_1x128_rowcol(a)",
                               "quant_128x128(out_proj)", "gemm_fwd(out_proj)"], world,
                              extra={"model_torch_ops_ms": round(torch_ms, 4),
                                     "note": "the activation and its gradient are the model's torch ops, not library "
                                             "calls; on this 1 % outlier-row workload the method itself reaches SQNR "
                                             "16.8-25.6 dB against the unquantized product (dx 19.3, d_w1 16.8), below "
                                             "the 25 dB single-linear bar"})


def run_chain_epilogue_quant(dev, steps, warmup, fp8_peak, hbm_peak, world):
    """Forward of two chained blockwise linears, y2 = (x W1^T) W2^T, at the
    toy FFN's sizes (tokens 4096, dim 2048, hidden 8192), with the hidden
    activation y1 quantized (rowwise for the next forward, colwise for its
    grad_weight) either by the stand-alone fused quantizer or in the epilogue
    of the GEMM that produces it (fp8bw_gemm_fwd_quant).  Weights are
    quantized once outside the timed calls."""
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B

    M_, D_, H_ = 4096, 2048, 8192
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    draw = lambda shape, std: (torch.randn(shape, generator=g, device=dev) * std).bfloat16()  # noqa: E731
    x, w1, w2 = draw((M_, D_), 1.0), draw((H_, D_), 0.02), draw((D_, H_), 0.02)
    xq, xs = B.alloc_quant_1x128_row(x)
    xqT, xsT = B.alloc_quant_1x128_col(x)
    w1q, _, w1s = B.alloc_quant_128x128(w1, False)
    w2q, _, w2s = B.alloc_quant_128x128(w2, False)
    B.fp8bw_quant_128x128(w1, w1q, None, w1s)
    B.fp8bw_quant_128x128(w2, w2q, None, w2s)
    y1 = torch.empty((M_, H_), dtype=torch.bfloat16, device=dev)
    y2 = torch.empty((M_, D_), dtype=torch.bfloat16, device=dev)
    q1, s1 = B.alloc_quant_1x128_row(y1)
    q1T, s1T = B.alloc_quant_1x128_col(y1)
    qx = lambda: B.fp8bw_quant_1x128_rowcol(x, xq, xs, xqT, xsT)  # noqa: E731
    separate = [("quant_1x128_rowcol(x)", qx),
                ("gemm_fwd(w1)", lambda: B.fp8bw_gemm_fwd(xq, xs, w1q, w1s, y1)),
                ("quant_1x128_rowcol(y1)", lambda: B.fp8bw_quant_1x128_rowcol(y1, q1, s1, q1T, s1T)),
                ("gemm_fwd(w2)", lambda: B.fp8bw_gemm_fwd(q1, s1, w2q, w2s, y2))]
    fused = [("quant_1x128_rowcol(x)", qx),
             ("gemm_fwd_quant(w1)", lambda: B.fp8bw_gemm_fwd_quant(xq, xs, w1q, w1s, y1, q1, s1, q1T, s1T)),
             ("gemm_fwd(w2)", lambda: B.fp8bw_gemm_fwd(q1, s1, w2q, w2s, y2))]
    out = {"workload": f"two chained blockwise linears, forward, tokens={M_} dim={D_} hidden={H_}, hidden activation "
                       "quantized rowwise and colwise; device-drawn N(0,1) x, N(0,0.02) weights, seed 1"}
    for name, kern in (("separate_quantizer", separate), ("epilogue_quantizer", fused)):
        for _ in range(warmup):
            for _, fn in kern:
                fn()
        B.fp8bw_sync_status()
        barrier(world)
        ms, per = time_kernels(kern, steps, torch.cuda.current_stream(dev))
        B.fp8bw_sync_status()
        out[name] = {"ms_per_step": round(max_over_ranks(world, ms, dev), 4),
                     "calls_us": {n: round(v * 1e3, 1) for n, v in per.items()}}
    out["saved_us"] = round(1e3 * (out["separate_quantizer"]["ms_per_step"] - out["epilogue_quantizer"]["ms_per_step"]),
                            1)
    del x, w1, w2, y1, y2
    torch.cuda.empty_cache()
    return out


# (M, N, K) rows of the grouped-mm microbenchmark of PR #3037, each at G = 1, 2, 4, 8.
MOE_TABLE_MNK = [(16384, 8192, 5120), (128000, 8192, 5120), (16384, 1536, 5120), (128000, 1536, 5120),
                 (16384, 2048, 7168), (128000, 2048, 7168)]


# (M, K, N) of the blockwise linear workloads: the dense one and the two large-token ones.
DENSE_TABLE_MKN = [(16384, 5120, 8192), (128000, 7168, 2048), (128000, 5120, 1536)]


def run_dense_table(dev, steps, warmup):
    """The blockwise-FP8 linear (six calls) over the dense and large-token
    workload shapes: per-kernel microseconds, forward (x and W quantization +
    fwd GEMM) and forward+backward microseconds, GEMM TFLOP/s.  One JSON line
    per shape; seeded device-side draws, timing only."""
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
    from mxfp8_precision_gemms_fp8bw_gb300.linear import BlockwiseLinearWorkspace

    for (M, K, N) in DENSE_TABLE_MKN:
        g = torch.Generator(device=dev)
        g.manual_seed(M + K + N)
        draw = lambda shape, std: (torch.randn(shape, generator=g, device=dev) * std).bfloat16()  # noqa: E731
        x, w, dy = draw((M, K), 1.0), draw((N, K), 0.02), draw((M, N), 1e-3)
        ws = BlockwiseLinearWorkspace(M, N, K, device=dev)
        kern = ws.kernels(x, w, dy)
        for _ in range(warmup):
            ws.step(x, w, dy)
        B.fp8bw_sync_status()
        ms, per = time_kernels(kern, steps, torch.cuda.current_stream(dev))
        B.fp8bw_sync_status()
        lu = linear_us(per, ["quant_1x128_rowcol(x)", "quant_128x128(W)", "gemm_fwd"])
        gemm_ms = sum(v for n, v in per.items() if n.startswith("gemm"))
        print(json.dumps({"table": "blockwise_linear", "M": M, "K": K, "N": N, **lu,
                          "kernels_us": {n: round(v * 1e3, 1) for n, v in per.items()},
                          "gemm_tflops": round(6 * M * N * K / (gemm_ms * 1e-3) / 1e12, 1),
                          "fwd_bwd_tflops": round(6 * M * N * K / (lu["fwd_bwd_us"] * 1e-6) / 1e12, 1)}),
              flush=True)
        del x, w, dy, ws, kern
        torch.cuda.empty_cache()
    return 0


def run_moe_table(dev, steps, warmup):
    """The MXFP8 grouped linear over the shapes of PR #3037's microbenchmark
    table, in its columns: forward (the fused row + column quantizations of x
    and W, which also produce the backward's colwise operands, and the
    grouped GEMM) and forward + backward (the whole six-call step) in
    microseconds.  One JSON line per
    shape; inputs are seeded N(0,1) / N(0,0.02) / N(0,1e-3) draws made on the
    device (timing only, no parity check), token groups of multiples of 32."""
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
    from mxfp8_precision_gemms_fp8bw_gb300 import inputs
    from mxfp8_precision_gemms_fp8bw_gb300.linear import MxMoEWorkspace

    for (M, N, K) in MOE_TABLE_MNK:
        for G in (1, 2, 4, 8):
            g = torch.Generator(device=dev)
            g.manual_seed(1000 * G + M % 1000 + N + K)
            draw = lambda shape, std: (torch.randn(shape, generator=g, device=dev) * std).bfloat16()  # noqa: E731
            x, w, dy = draw((M, K), 1.0), draw((G, N, K), 0.02), draw((M, N), 1e-3)
            sizes = inputs.moe_group_sizes(np.random.default_rng(G), M, G)
            ge = torch.from_numpy(np.cumsum(sizes).astype(np.int32)).to(dev)
            ws = MxMoEWorkspace(M, N, K, G, device=dev)
            kern = ws.kernels(x, w, dy, ge)
            for _ in range(warmup):
                ws.step(x, w, dy, ge)
            B.fp8bw_sync_status()
            ms, per = time_kernels(kern, steps, torch.cuda.current_stream(dev))
            B.fp8bw_sync_status()
            lu = linear_us(per, ["mx_quant_1x32_rowcol(x)", "mx_quant_1x32_rowcol(W)", "mx_grouped_fwd"])
            print(json.dumps({"table": "mxfp8_grouped_mm", "M": M, "N": N, "K": K, "G": G, **lu,
                              "fwd_bwd_tflops": round(6 * M * N * K / (lu["fwd_bwd_us"] * 1e-6) / 1e12, 1)}),
                  flush=True)
            del x, w, dy, ws, kern
            torch.cuda.empty_cache()
    return 0


def load_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu
    summary, if the kernel's sources still hash to what was profiled; else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)["kernels"].get(kernel)
        if entry is None:
            return None
        from mxfp8_precision_gemms_fp8bw_gb300 import build as _b
        h = hashlib.sha256()
        for name in entry["sources"]:
            with open(os.path.join(_b.CSRC, name), "rb") as f:
                h.update(f.read())
        return entry["bytes"] if h.hexdigest()[:16] == entry["hash"] else None
    except (OSError, ValueError, KeyError):
        return None


def run_section(args, world, local):
    """One workload's step alone (see --section): a single JSON line."""
    import torch

    from mxfp8_precision_gemms_fp8bw_gb300 import binding as B

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.lib(build_if_missing=True)
    peaks = load_peaks()
    fp8_peak, hbm = peaks["bf16"] * FP8_OVER_BF16, peaks["hbm_gbs"]
    steps, warmup = args.steps, args.warmup
    if args.section == "dense":
        from mxfp8_precision_gemms_fp8bw_gb300.linear import BlockwiseLinearWorkspace
        t = dense_inputs()
        x, w, dy = t.x.to(dev), t.w.to(dev), t.dy.to(dev)
        ws = BlockwiseLinearWorkspace(M, N, K, device=dev)
        kern = ws.kernels(x, w, dy)
        for _ in range(warmup):
            ws.step(x, w, dy)
        B.fp8bw_sync_status()
        ms, per = time_kernels(kern, steps, torch.cuda.current_stream(dev))
        B.fp8bw_sync_status()
        sec = section_from_times(WORKLOAD, per, ws.algorithmic(), 6 * M * N * K, ms, steps, fp8_peak, hbm,
                                 ["quant_1x128_rowcol(x)", "quant_128x128(W)", "gemm_fwd"], world)
    elif args.section in ("large0", "large1"):
        sec = run_large_token(dev, int(args.section[-1]), steps, warmup, fp8_peak, hbm, world)
    elif args.section == "ffn":
        sec = run_ffn(dev, steps, warmup, fp8_peak, hbm, world)
    elif args.section == "chain":
        sec = run_chain_epilogue_quant(dev, steps, warmup, fp8_peak, hbm, world)
    else:
        sec = run_moe(dev, steps, warmup, fp8_peak, hbm, world, dense=args.section == "mxdense")
    print(json.dumps({"section": args.section, **sec}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-moe", action="store_true", help="skip the MXFP8 sections (MoE and dense)")
    ap.add_argument("--section", choices=["dense", "large0", "large1", "ffn", "chain", "moe", "mxdense"],
                    help="run only this workload's step (--warmup untimed, --steps timed) and print its section as "
                         "one JSON line: for profiling one kernel on one workload")
    ap.add_argument("--tables", action="store_true",
                    help="instead of the bench line, time the blockwise linear over the dense and large-token "
                         "shapes and the MXFP8 grouped linear over the shapes of the grouped-mm microbenchmark "
                         "table (one JSON line per shape)")
    args = ap.parse_args()
    if not args.section:
        args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.impl == "reference":
        # Rank 0 alone times the CPU oracle; the other ranks exit without work
        # (no process group: nothing is exchanged).
        world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
        return run_reference(args, world, rank)
    world, rank, local = dist_setup(args.gpus)
    if args.section:
        return run_section(args, world, local)
    if args.tables:
        import torch
        torch.cuda.set_device(local)
        from mxfp8_precision_gemms_fp8bw_gb300 import binding as B
        B.lib(build_if_missing=True)
        dev = torch.device("cuda", local)
        run_dense_table(dev, min(args.steps, 20), args.warmup)
        return run_moe_table(dev, min(args.steps, 20), args.warmup)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
