#!/usr/bin/env python3
"""Benchmark of the forward linear-layer family on one GB300 per rank.

A step is one call of the fused SwiGLU down projection with binary16
weights, ``lin_matmul_residual_swiglu_a_w16`` at M=16384 tokens, N=2048,
K=8192 (the scaled-up workload; it runs every step of the hot path: TMA
staging, the SwiGLU transform, binary16 rounding, the tcgen05 contraction and
the residual epilogue). Its inputs (1.3 GB) are far larger than the 129 MB
L2, so no flush is needed between steps.

Printed: one JSON line on rank 0 with the metric (TFLOP/s = 2MNK / time),
the roofline of the GEMM kernel, the end-to-end figure (host buffers, copies
inside the timed region), the oracle's CPU baseline, SM clocks sampled during
the timed region, and a per-workload table for the four small transformer
shapes (each timed cold, after an L2 flush, and warm, back to back).

``--impl reference`` times the fp64 CPU oracle instead (rank 0 only), each
step a bounded sample of rows of the same workload.

Multi-GPU: one process per GPU, under torchrun, or started by ``--gpus N``
itself when no launcher set WORLD_SIZE; the path shards over tokens with no
exchange, so every rank runs its own replica of the workload ("replicas
only", weak scaling) and value = all ranks' FLOPs / the slowest rank's time.

``--measure-peaks`` prints this GPU's cuBLAS TF32 / binary16 / bfloat16
peaks (the TF32 one, recorded in profiles/tensor_peaks.txt, is the roofline
peak of the f32 forms).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from transformer_linear_layer_tcgen05_gb300 import workloads as wl  # noqa: E402

METRIC = "TFLOP/s per linear-form GEMM on 1 GB300 and % of tensor-core roofline"
HEADLINE = "ffn_down_swiglu_w16_16k"
SMALL = ("attn_proj_f32", "ffn_up_residual_f32", "ffn_down_swiglu_f32", "lm_head_w16")
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense rates relative to bf16 (2.25 PFLOP/s): f16 1.0, tf32 1.1/2.25.
NOMINAL_RATIO = {"f16": 1.0, "tf32": 1.1 / 2.25}


# ----------------------------------------------------------------- helpers

def recorded_tensor_peaks() -> dict:
    """The TF32 peaks (burst, sustained; TFLOP/s) measured on this machine's
    GB300s by ``--measure-peaks`` and recorded in profiles/tensor_peaks.txt
    (empty if absent)."""
    p = os.path.join(ROOT, "profiles", "tensor_peaks.txt")
    out = {}
    if os.path.exists(p):
        with open(p) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 2 and not line.startswith("#") and \
                        parts[0] in ("tf32_tflops", "tf32_tflops_sustained"):
                    out[parts[0]] = float(parts[1])
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        src = "measured"
    else:
        d, src = dict(FALLBACK_PEAKS), "fallback"
    d.update(recorded_tensor_peaks())
    return d, src


# The sources the dominant kernel (the clustered SwiGLU GEMM) is compiled
# from: its translation unit and every header it includes.
DOMINANT_KERNEL_SOURCES = ("lin_kernels_cluster_swiglu.cu", "lin_gemm_cluster.cuh",
                           "lin_common.cuh", "lin_ptx.cuh", "lin_internal.h")


def kernel_source_hash() -> str:
    """Hash of the dominant kernel's sources (a recorded DRAM figure is
    valid only for the code it was captured on)."""
    csrc = os.path.join(ROOT, "transformer_linear_layer_tcgen05_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(DOMINANT_KERNEL_SOURCES):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash()
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload \
                    and parts[1] == want:
                return int(parts[2])
    return None


def kernel_label(w: wl.Workload) -> str:
    """Name of the kernel the library dispatches for workload w (the
    binary16 forms run the clustered kernel: clusters of 4 from N >= 1024,
    pairs from N >= 512, else single CTAs; single CTAs too where X is
    rounded to binary16 by a pre-pass, from N >= 2048 for the forms that
    read X)."""
    if w.form.endswith("_w16"):
        cols = w.K if wl.form_is_t(w.form) else w.N   # output columns
        cn = os.environ.get("LIN_F16_KERNEL") or ("4" if cols >= 1024 else "2" if cols >= 512 else "1")
        if not os.environ.get("LIN_F16_KERNEL") and "swiglu_a" not in w.form and cols >= 2048:
            return "lin_cvt_f16_kernel + lin_gemm_cluster_kernel (BN=256, single CTAs, A by TMA)"
        if cn == "tile":
            return "lin_gemm_kernel (per-tile, BN=128)"
        return f"lin_gemm_cluster_kernel (BN=256, cluster {cn} along N)"
    return "lin_gemm_kernel (per-tile, BN=128, TF32)"


def mma_dtype(form: str) -> str:
    return "f16" if form.endswith("_w16") else "tf32"


def tensor_peak(dtype: str, peaks: dict, sustained: bool = False):
    """(peak TFLOP/s, where it comes from) of the contraction's own dtype:
    the measured TF32 peak for the f32 forms where one is recorded, else the
    measured bfloat16 peak times the nominal ratio (binary16: 1.0)."""
    key = f"{dtype}_tflops" + ("_sustained" if sustained else "")
    if dtype == "tf32" and key in peaks:
        return peaks[key], "measured tf32 (cuBLAS, profiles/tensor_peaks.txt)"
    bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return bf16 * NOMINAL_RATIO[dtype], f"bf16 x nominal {dtype}/bf16 ratio {NOMINAL_RATIO[dtype]:.3g}"


def roofline(w: wl.Workload, peaks: dict, sustained: bool = False):
    """(bound, roofline TFLOP/s, tensor peak TFLOP/s, HBM GB/s) of workload w:
    min(peak FLOP/s, algorithmic bytes / HBM bandwidth * FLOP/byte)."""
    tpeak = tensor_peak(mma_dtype(w.form), peaks, sustained)[0]
    hbm = peaks["hbm_gbs"]
    nbytes = wl.input_bytes(w.form, w.M, w.N, w.K)
    mem_tflops = w.flops / nbytes * hbm / 1e3
    if mem_tflops < tpeak:
        return "hbm", mem_tflops, tpeak, hbm
    return "tensor", tpeak, tpeak, hbm


class ClockSampler:
    """SM clock, power and clock-event reasons sampled during a timed region.

    Read-only NVML queries (libnvidia-ml through ctypes: the SM clock, its
    maximum, the power draw and the active clock-event reasons) every
    `period_s` in a thread, so that even a timed region of a few milliseconds
    holds several samples; where NVML cannot be loaded, nvidia-smi's own
    200 ms loop. Nothing here sets any GPU state. A sample is (host time,
    SM MHz, max SM MHz, power W, set of reason names)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # nvmlClocksEventReason* bits (nvml.h) of the reasons the bench reports
    REASON_BITS = ((0x8, "hw_slowdown"), (0x40, "hw_thermal_slowdown"),
                   (0x20, "sw_thermal_slowdown"), (0x4, "sw_power_cap"))
    NVML_CLOCK_SM = 1

    def __init__(self, gpu_id: str | None, period_s: float = 0.002):
        self.gpu_id = gpu_id          # "GPU-<uuid>", or None for the first GPU
        self.period_s = period_s
        self.samples = []
        self.source = None
        self.proc = None
        self.thread = None
        self._stop = threading.Event()

    # -- NVML (read-only queries)
    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        dev = ctypes.c_void_p()
        if self.gpu_id:
            rc = lib.nvmlDeviceGetHandleByUUID(self.gpu_id.encode(), ctypes.byref(dev))
        else:
            rc = lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(dev))
        if rc != 0:
            lib.nvmlShutdown()
            raise OSError("no NVML handle for the device")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, dev, reasons_fn

    def _nvml_loop(self, lib, dev, reasons_fn):
        import ctypes
        sm, smax, mw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        lib.nvmlDeviceGetMaxClockInfo(dev, self.NVML_CLOCK_SM, ctypes.byref(smax))
        try:
            while not self._stop.is_set():
                t = time.time()
                ok = lib.nvmlDeviceGetClockInfo(dev, self.NVML_CLOCK_SM, ctypes.byref(sm)) == 0
                pw = lib.nvmlDeviceGetPowerUsage(dev, ctypes.byref(mw)) == 0
                rok = reasons_fn(dev, ctypes.byref(rs)) == 0
                if ok:
                    names = frozenset(n for b, n in self.REASON_BITS if rok and rs.value & b)
                    self.samples.append((t, float(sm.value), float(smax.value) or None,
                                         mw.value / 1000.0 if pw else None, names))
                time.sleep(self.period_s)
        finally:
            lib.nvmlShutdown()

    # -- nvidia-smi fallback
    def _smi_read(self):
        for line in self.proc.stdout:
            self.samples.append(self.parse_smi_row(time.time(), line))

    @classmethod
    def parse_smi_row(cls, t: float, line: str):
        f = [x.strip() for x in line.split(",")]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        if len(f) < 9:
            return (t, None, None, None, frozenset())
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        active = frozenset(n for n, v in zip(names, f[5:9]) if v.lower() == "active")
        return (t, num(f[1]), num(f[2]), num(f[3]), active)

    def start(self):
        try:
            lib, dev, reasons_fn = self._nvml_open()
            self.source = f"NVML every {self.period_s * 1e3:.0f} ms"
            self.thread = threading.Thread(target=self._nvml_loop, args=(lib, dev, reasons_fn),
                                           daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            pass
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.source = "nvidia-smi every 200 ms"
        self.thread = threading.Thread(target=self._smi_read, daemon=True)
        self.thread.start()

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        """Median SM clock, its maximum, the reasons seen and the peak power
        over the samples taken between host times t0 and t1 (all samples when
        none fell inside)."""
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        used = inside if inside else list(self.samples)
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "samples_in_timed_region": 0, "source": self.source,
                    "note": "no clock source available"}
        sm = [s[1] for s in used if s[1] is not None]
        smax = [s[2] for s in used if s[2] is not None]
        power = [s[3] for s in used if s[3] is not None]
        reasons = sorted(set().union(*(s[4] for s in used)))
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons,
                "power_w_max": max(power) if power else None,
                "samples": len(used), "samples_in_timed_region": len(inside),
                "source": self.source}


def oracle_threads() -> int:
    """Host threads the oracle's contraction runs on (its OpenMP row loop)."""
    import oracle
    return oracle.contraction_threads()


def cpu_baseline(w: wl.Workload, inputs: dict, budget_s: float = 12.0, chunk: int = 64):
    """Time the fp64 oracle, as it stands, on consecutive row chunks of the
    workload until about `budget_s` seconds of CPU work are done."""
    import numpy as np
    import oracle
    rows_done = 0
    t0 = time.perf_counter()
    start = 0
    while True:
        rows = np.arange(start, min(start + chunk, w.M))
        oracle.reference(w.form, inputs, rows=rows)
        rows_done += len(rows)
        start = (start + chunk) % w.M
        if time.perf_counter() - t0 >= budget_s or rows_done >= w.M:
            break
    dt = time.perf_counter() - t0
    flops = 2.0 * rows_done * w.N * w.K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(),
            "kind": "oracle",
            "sample": f"{rows_done} of {w.M} rows of {w.name} ({w.describe()}), "
                      f"fp64 C triple-loop oracle incl. normaliser, {dt:.1f} s"}


# ----------------------------------------------------------------- reference arm

def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's value (with times: the slowest rank's),
    by an all-reduce on `device` (cuda under NCCL, cpu under gloo); the value
    itself without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replicas_value(world: int, flops_per_rank: float, ms_max: float) -> float:
    """Whole-job TFLOP/s of `world` replicas of one workload: every rank's
    FLOPs over the slowest rank's time (the path shards over tokens with no
    exchange, so each rank runs the whole workload: weak scaling)."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def run_reference(args, rank: int):
    if rank != 0:
        world = os.environ.get("WORLD_SIZE", "?")
        print(f"bench: rank {rank} of {world}: the reference arm runs on rank 0 only",
              file=sys.stderr, flush=True)
        return
    import numpy as np
    import oracle
    w = wl.WORKLOADS_BY_NAME[args.workload]
    # Only the sampled rows are drawn in full size where needed: the generator
    # draws the whole workload, then the oracle reads a row sample per step.
    inputs = wl.generate_workload(w)
    rows_per_step = args.ref_rows
    starts = [(i * rows_per_step) % w.M for i in range(args.warmup + args.steps)]
    for s in starts[:args.warmup]:
        oracle.reference(w.form, inputs, rows=np.arange(s, min(s + rows_per_step, w.M)))
    t0 = time.perf_counter()
    nrows = 0
    for s in starts[args.warmup:]:
        rows = np.arange(s, min(s + rows_per_step, w.M))
        oracle.reference(w.form, inputs, rows=rows)
        nrows += len(rows)
    dt = time.perf_counter() - t0
    value = 2.0 * nrows * w.N * w.K / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / max(args.steps, 1) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "form": w.form, "M": w.M, "N": w.N, "K": w.K,
                   "sample_rows_per_step": rows_per_step},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle",
                         "cores": oracle_threads(),
                         "sample": f"{rows_per_step} rows of {w.M} per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- our arm

def device_inputs(inputs: dict):
    import numpy as np
    import torch
    return {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).cuda()
            for k, v in inputs.items()}


def time_small(w: wl.Workload, iters: int, flush_buf):
    """Cold (L2 flushed before each call) and warm (graph of back-to-back
    calls) kernel times of a small workload, in microseconds, plus its error
    is not computed here (the GPU tests cover parity)."""
    import torch
    from transformer_linear_layer_tcgen05_gb300 import lin
    d = device_inputs(wl.generate_workload(w))
    Y = torch.empty(wl.output_shape(w.form, w.M, w.N, w.K), dtype=torch.float32, device="cuda")
    if wl.form_is_swiglu_bwd(w.form):   # two outputs: dGATE, dUP
        Y = (Y, torch.empty_like(Y))
    stream = torch.cuda.current_stream()
    for _ in range(5):
        lin.run_form(w.form, d, Y)
    torch.cuda.synchronize()
    cold = []
    for _ in range(iters):
        flush_buf.fill_(1.0)           # evicts L2 and keeps the GPU busy while we enqueue
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        lin.run_form(w.form, d, Y)
        e1.record(stream)
        e1.synchronize()
        cold.append(e0.elapsed_time(e1) * 1e3)
    # warm: capture `reps` calls into a CUDA graph and replay it
    reps = 20
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            for _ in range(reps):
                lin.run_form(w.form, d, Y)
    stream.wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    warm = []
    for _ in range(max(3, iters // 10)):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        warm.append(e0.elapsed_time(e1) * 1e3 / reps)
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    del g
    return statistics.median(cold), statistics.median(warm)


def time_lm_head_loss(iters: int, flush_buf, peaks: dict) -> dict:
    """lm_head_w16's shape (512 x 16384 x 768) through
    lin_lm_head_cross_entropy_w16 (label smoothing 0.1, z-loss 1e-4), cold
    and warm like the small table. Algorithmic bytes: X, W16, targets in,
    dLogits and the losses out."""
    import numpy as np
    import torch
    from transformer_linear_layer_tcgen05_gb300 import lin
    w = wl.WORKLOADS_BY_NAME["lm_head_w16"]
    d = device_inputs(wl.generate_workload(w))
    rng = np.random.default_rng(77)
    t = torch.from_numpy(rng.integers(0, w.N, size=w.M).astype(np.int32)).cuda()
    DL = torch.empty((w.M, w.N), device="cuda")
    losses = torch.empty((w.M,), device="cuda")
    total = torch.empty((1,), device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        lin.lin_lm_head_cross_entropy_w16(d["X"], d["W16"], t, DL, losses, total, 0.1, 1e-4,
                                          1.0 / w.M)
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    cold = []
    for _ in range(iters):
        flush_buf.fill_(1.0)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        cold.append(e0.elapsed_time(e1) * 1e3)
    reps = 20
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(stream)
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            for _ in range(reps):
                call()
    stream.wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    warm = []
    for _ in range(max(3, iters // 10)):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        warm.append(e0.elapsed_time(e1) * 1e3 / reps)
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    del g
    nbytes = w.M * w.K * 4 + w.K * w.N * 2 + w.M * 4 + w.M * w.N * 4 + w.M * 4
    bf16 = peaks["bf16_tflops"]
    r = min(bf16, w.flops / nbytes * peaks["hbm_gbs"] / 1e3)
    c, wm = statistics.median(cold), statistics.median(warm)
    return {"workload": "lm_head_cross_entropy_w16", "M": w.M, "N": w.N, "K": w.K,
            "alpha": 0.1, "beta": 1e-4, "bound": "hbm" if r < bf16 else "tensor",
            "roofline_tflops": r, "cold_us": c, "cold_tflops": w.flops / c / 1e6,
            "cold_frac": w.flops / c / 1e6 / r, "warm_us": wm, "warm_tflops": w.flops / wm / 1e6,
            "warm_frac": w.flops / wm / 1e6 / r}


def time_gate_up(iters: int, flush_buf, peaks: dict, M: int = 16384) -> dict:
    """The producer of the 16k SwiGLU workload's GATE and UP through
    lin_gate_up_w16: X [M, 2048] f32, W_gate and W_up [2048, 8192] binary16
    (2 x 550 GFLOP at M = 16384), timed cold (inputs above L2 anyway) and
    warm. A smaller M serves profiling captures."""
    import numpy as np
    import torch
    from transformer_linear_layer_tcgen05_gb300 import lin
    N, K = 8192, 2048
    g = wl.generate("matmul_w16", M, N, K, seed=1020)
    wu = wl.generate("matmul_w16", 1, N, K, seed=1021)["W16"]
    X = torch.from_numpy(g["X"]).cuda()
    WG = torch.from_numpy(g["W16"].view(np.int16)).cuda()
    WU = torch.from_numpy(wu.view(np.int16)).cuda()
    G = torch.empty((M, N), device="cuda")
    U = torch.empty((M, N), device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        lin.lin_gate_up_w16(X, WG, WU, G, U)

    def separate():   # the two products it replaces, one lin_matmul_w16 each
        lin.lin_matmul_w16(X, WG, G)
        lin.lin_matmul_w16(X, WU, U)

    def timed_us(fn):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3

    # The two ways alternate call by call (medians of each), so that neither
    # runs in a later, hotter part of the table than the other: under the
    # power cap the clock falls as the 16k-token tables go on.
    for _ in range(3):
        separate()
        call()
    torch.cuda.synchronize()
    sep_times, times = [], []
    for _ in range(max(5, iters // 5)):
        sep_times.append(timed_us(separate))
        times.append(timed_us(call))
    assert lin.lin_get_device_status() == lin.LIN_SUCCESS
    sep_us = statistics.median(sep_times)
    us = statistics.median(times)
    flops = 2 * 2 * M * N * K
    nbytes = M * K * 4 + 2 * K * N * 2 + 2 * M * N * 4
    bf16 = peaks["bf16_tflops"]
    r = min(bf16, flops / nbytes * peaks["hbm_gbs"] / 1e3)
    return {"workload": "ffn_gate_up_w16_16k", "form": "gate_up_w16", "M": M, "N": N, "K": K,
            "two_matmul_w16_us": sep_us,
            "bound": "hbm" if r < bf16 else "tensor", "roofline_tflops": r, "cold_us": us,
            "cold_tflops": flops / us / 1e6, "cold_frac": flops / us / 1e6 / r, "warm_us": us,
            "warm_tflops": flops / us / 1e6, "warm_frac": flops / us / 1e6 / r}


def run_ours(args, rank: int, world: int):
    import numpy as np
    import torch
    from transformer_linear_layer_tcgen05_gb300 import build as _build
    from transformer_linear_layer_tcgen05_gb300 import lin

    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    _build.build_library()
    lin.lib()
    peaks, peak_src = load_peaks()
    w = wl.WORKLOADS_BY_NAME[args.workload]
    if args.m is not None:
        import dataclasses
        w = dataclasses.replace(w, M=args.m)

    def barrier():
        if dist is not None:
            dist.barrier()

    # ---- inputs resident in HBM before the timed region
    host = wl.generate_workload(w)
    d = device_inputs(host)
    Y = torch.empty(wl.output_shape(w.form, w.M, w.N, w.K), dtype=torch.float32, device="cuda")
    if wl.form_is_swiglu_bwd(w.form):   # two outputs: dGATE, dUP
        Y = (Y, torch.empty_like(Y))
    stream = torch.cuda.current_stream()

    def step():
        lin.run_form(w.form, d, Y)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if lin.lin_get_device_status() != lin.LIN_SUCCESS:
        raise RuntimeError("device status after warm-up is not LIN_SUCCESS")
    # kernels one step launches (2 when the persistent launch splits its last
    # round along K: the GEMM, then the sum of the tail's partial tiles)
    step()
    kernels_per_step, workspace_bytes = lin.lin_last_launch_info()
    torch.cuda.synchronize()

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        gpu_id = None
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.5)

    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    h0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    e1.synchronize()
    h1 = time.time()
    torch.cuda.synchronize()
    barrier()
    sampler.stop()
    ms = e0.elapsed_time(e1) / max(args.steps, 1)
    status = lin.lin_get_device_status()
    if status != lin.LIN_SUCCESS:
        raise RuntimeError(f"device status {lin.STATUS.get(status, status)} after timed region")

    ms_max = max_over_ranks(ms, dist, "cuda")
    value = replicas_value(world, w.flops, ms_max)
    kernel_tflops = w.flops / (ms * 1e-3) / 1e12

    # ---- end to end through the public API: pinned host buffers, H2D of the
    # step's inputs, the call, D2H of Y, all inside the timed region. The
    # forward forms take the host-operand entry point (the library's own
    # copies, in row blocks overlapped with the GEMMs); the others copy with
    # torch around the device entry point.
    e2e_steps = 0 if args.no_e2e else max(3, min(args.steps, args.e2e_steps))
    pinned = {k: torch.from_numpy(v.view(np.int16) if v.dtype == np.uint16 else v).pin_memory()
              for k, v in host.items()}
    outs = Y if isinstance(Y, tuple) else (Y,)
    y_host = [torch.empty(o.shape, dtype=torch.float32).pin_memory() for o in outs]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(y.numel() * 4 for y in y_host)

    host_api = w.form in lin.HOST_FORM_FUNCS

    def e2e_step():
        if host_api:
            lin.run_form_host(w.form, pinned, y_host[0])
            return
        for k, t in pinned.items():
            d[k].copy_(t, non_blocking=True)
        lin.run_form(w.form, d, Y)
        for yh, o in zip(y_host, outs):
            yh.copy_(o, non_blocking=True)

    for _ in range(args.e2e_warmup if e2e_steps else 0):   # untimed calls first
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    f1.record(stream)
    f1.synchronize()
    e2e_ms = f0.elapsed_time(f1) / max(e2e_steps, 1)
    e2e_max = max_over_ranks(e2e_ms, dist, "cuda")
    e2e_value = replicas_value(world, w.flops, e2e_max) if e2e_steps else None
    del pinned, y_host

    # ---- roofline of the step's GEMM; achieved = the step's FLOPs over the
    # whole step time (with a split tail that includes the tail-sum kernel).
    # A timed region of seconds of back-to-back launches runs under the power
    # cap, so it is compared with the sustained peak; a short one with the
    # burst peak.
    timed_s = ms * args.steps / 1e3
    sustained = timed_s > 1.0
    bound, roof, tpeak, hbm = roofline(w, peaks, sustained=sustained)
    traffic = recorded_traffic(w.name)
    peak_txt = tensor_peak(mma_dtype(w.form), peaks, sustained)[1]
    roof_obj = {"bound": bound, "achieved": kernel_tflops, "peak": roof, "unit": "TFLOP/s",
                "frac": kernel_tflops / roof, "traffic": traffic,
                "peak_source": f"{peak_src} peaks: {peak_txt} "
                               f"({'sustained: timed region %.1f s' % timed_s if sustained else 'burst: timed region %.2f s' % timed_s})",
                "peak_burst": roofline(w, peaks, sustained=False)[1],
                "peak_sustained": roofline(w, peaks, sustained=True)[1],
                "kernel": kernel_label(w) + (" + lin_split_reduce_kernel (split tail)"
                                             if kernels_per_step > 1 else ""),
                "timed": "whole step (all kernels of the call)",
                "workspace_bytes": workspace_bytes,
                "algorithmic_bytes": wl.input_bytes(w.form, w.M, w.N, w.K),
                "algorithmic_flops": w.flops}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": w.name, "form": w.form, "M": w.M, "N": w.N, "K": w.K,
                   "l2": f"inputs {wl.input_bytes(w.form, w.M, w.N, w.K) / 1e9:.2f} GB > L2, no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof_obj,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "call": (f"lin_{w.form}_host (pinned host buffers)" if host_api
                         else f"torch copies + lin_{w.form}")},
        "gpu_launches": args.steps * kernels_per_step,
        "clocks": sampler.summary(h0, h1),
    }

    tables = set(args.tables.split(","))
    if rank == 0 and not args.no_small:
        flush = torch.empty(int(2 * L2_BYTES // 4), dtype=torch.float32, device="cuda")
    if rank == 0 and not args.no_small and "workloads" in tables:
        table = []
        for name in SMALL:
            sw = wl.WORKLOADS_BY_NAME[name]
            cold_us, warm_us = time_small(sw, args.small_iters, flush)
            b, r, tp, _ = roofline(sw, peaks)
            table.append({"workload": name, "form": sw.form, "M": sw.M, "N": sw.N, "K": sw.K,
                          "bound": b, "roofline_tflops": r,
                          "tensor_peak_source": tensor_peak(mma_dtype(sw.form), peaks)[1],
                          "cold_us": cold_us, "cold_tflops": sw.flops / cold_us / 1e6,
                          "cold_frac": sw.flops / cold_us / 1e6 / r,
                          "warm_us": warm_us, "warm_tflops": sw.flops / warm_us / 1e6,
                          "warm_frac": sw.flops / warm_us / 1e6 / r})
        line["workloads"] = table
    if rank == 0 and not args.no_small and "backward" in tables:
        # the backward products of the same layers, timed the same way
        table = []
        for sw in wl.BACKWARD_WORKLOADS:
            cold_us, warm_us = time_small(sw, args.small_iters, flush)
            b, r, tp, _ = roofline(sw, peaks)
            table.append({"workload": sw.name, "form": sw.form, "M": sw.M, "N": sw.N, "K": sw.K,
                          "bound": b, "roofline_tflops": r,
                          "tensor_peak_source": tensor_peak(mma_dtype(sw.form), peaks)[1],
                          "cold_us": cold_us, "cold_tflops": sw.flops / cold_us / 1e6,
                          "cold_frac": sw.flops / cold_us / 1e6 / r,
                          "warm_us": warm_us, "warm_tflops": sw.flops / warm_us / 1e6,
                          "warm_frac": sw.flops / warm_us / 1e6 / r})
        line["backward"] = table
    if rank == 0 and not args.no_small and "loss" in tables:
        line["loss"] = [time_lm_head_loss(args.small_iters, flush, peaks)]
    if rank == 0 and not args.no_small and "gate_up" in tables:
        line["gate_up"] = [time_gate_up(args.small_iters, flush, peaks, M=args.gate_up_m)]
    if rank == 0 and not args.no_small:
        del flush
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, host, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def launch_command(nproc: int, argv: list[str], port: int) -> list[str]:
    """The command that re-runs this script as `nproc` ranks of one node
    (torch.distributed.run on 127.0.0.1), with the same arguments."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={nproc}", "--master-addr", "127.0.0.1",
            "--master-port", str(port), os.path.abspath(__file__), *argv]


def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def measure_peaks(seconds: float = 3.0) -> dict:
    """Dense tensor-core peaks of this GPU as cuBLAS reaches them through
    torch.matmul at 8192^3 (2 N^3 FLOPs): TF32 (float32 with TF32 allowed),
    binary16 and bfloat16; each the best of 10 single calls (burst) and the
    rate of back-to-back calls over `seconds` (sustained), CUDA events on the
    current stream, with SM clocks sampled meanwhile."""
    import torch
    n = 8192
    flops = 2.0 * n ** 3
    out = {"how": f"torch.matmul {n}^3 (2*N^3): best of 10 (burst) and back to back for "
                  f"{seconds:.0f} s (sustained); CUDA events", "torch": torch.__version__,
           "gpu_name": torch.cuda.get_device_name()}
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        for name, dt in (("tf32", torch.float32), ("f16", torch.float16),
                         ("bf16", torch.bfloat16)):
            a = torch.randn(n, n, device="cuda").to(dt)
            b = torch.randn(n, n, device="cuda").to(dt)
            for _ in range(3):
                torch.matmul(a, b)
            torch.cuda.synchronize()
            best = float("inf")
            for _ in range(10):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                torch.matmul(a, b)
                e1.record()
                e1.synchronize()
                best = min(best, e0.elapsed_time(e1) * 1e-3)
            iters = max(1, int(seconds / best))
            sampler = ClockSampler(None, period_s=0.01)
            sampler.start()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            h0 = time.time()
            e0.record()
            for _ in range(iters):
                torch.matmul(a, b)
            e1.record()
            e1.synchronize()
            h1 = time.time()
            sampler.stop()
            sus = e0.elapsed_time(e1) * 1e-3 / iters
            out[f"{name}_tflops"] = flops / best / 1e12
            out[f"{name}_tflops_sustained"] = flops / sus / 1e12
            out[f"{name}_clocks_sustained"] = sampler.summary(h0, h1)
            del a, b
            torch.cuda.empty_cache()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000,
                    help="timed steps (about 2 s at the default workload, so that the "
                         "nvidia-smi clock samples fall inside the timed region)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=[w.name for w in wl.WORKLOADS + wl.BACKWARD_WORKLOADS])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-warmup", type=int, default=30,
                    help="untimed end-to-end calls before the timed ones")
    ap.add_argument("--small-iters", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=16)
    ap.add_argument("--no-small", action="store_true")
    ap.add_argument("--tables", default="workloads,backward,loss,gate_up",
                    help="comma-separated tables to run besides the headline")
    ap.add_argument("--gate-up-m", type=int, default=16384,
                    help="M of the gate/up table (a smaller M for profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--m", type=int, default=None,
                    help="override M (tokens) of the workload, e.g. a small case for ncu")
    ap.add_argument("--measure-peaks", action="store_true",
                    help="print the TF32, binary16 and bfloat16 cuBLAS peaks of this GPU "
                         "as one JSON line and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.measure_peaks:
        print(json.dumps(measure_peaks()), flush=True)
        return

    # --gpus N outside a launcher: start N ranks on this node, one per GPU
    # (each runs its own replica; rank 0 prints the line) and exit with
    # their status.
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(subprocess.call(launch_command(args.gpus, sys.argv[1:], _free_port())))

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
