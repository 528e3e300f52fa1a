#!/usr/bin/env python
"""Throughput of INT8 conv2d forward propagation (int32 results) on GB300.

One step = one full conv_fprop of the workload (filter repack kernel + the
tcgen05 implicit-GEMM kernel, which computes the output with bias/ReLU fused
when the workload asks for them).  Default workload: N=32, C=256, 56x56 image,
K=256, 3x3 filter, stride 1, padding 1, NHWC image / KRSC filter / NHWC output.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Throughput is 2*N*K*P*Q*C*R*S / time in
TOPS.  Inputs stay resident in HBM; successive steps rotate over several
input/output sets whose total exceeds the 129 MB L2, so every step starts
with cold caches.  Under torchrun each rank runs its own copy of the workload
(weak scaling, no collective on the data path); the elapsed time is the max
over ranks.  ``--impl reference`` times the CPU oracle on the host cores
instead (rank 0 only).

The line's ``workloads`` map holds one record per workload of the
specification (the five shapes, ``--workloads``), each over ``--launches``
launches with a cold L2: the step and the convolution call alone, as the
average of back-to-back launches over rotating sets (the large workloads) or
the median of launches each timed by its own events after a 258 MiB write
(the small ones); the isolated medians beside them; the step with a warm L2;
and a roofline per workload.  The headline ``roofline.kernel_ms`` is the
convolution call of the headline workload's record.  ``int8_routes`` holds
the measured dense rates of the int8-capable instruction routes
(conv_measure_peak_rates).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "INT8 conv fprop TOPS (2NKPQCRS/s) and % of GB300 dense INT8 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DOMINANT_KERNEL_SRC = os.path.join(ROOT, "int8_conv2d_fprop_gb300", "csrc", "igemm.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "igemm_traffic.json")
L2_BYTES = 129 * 1024 * 1024
ALL_WORKLOADS_DEFAULT = ("c1_tiny_nchw", "c2_s2_nhwc", "c3_3x3_large", "c4_1x1_bias_relu", "c5_7x1_dilated_conv")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3_3x3_large", choices=sorted(synth.CONFIGS))
    ap.add_argument("--workloads", default=",".join(ALL_WORKLOADS_DEFAULT),
                    help="comma-separated workloads timed one by one into the line's 'workloads' map "
                         "(empty: none)")
    ap.add_argument("--launches", type=int, default=60,
                    help="event-timed launches behind each median of the 'workloads' map (>= 50)")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-peak-probe", action="store_true",
                    help="skip the measured instruction-route rates (conv_measure_peak_rates)")
    ap.add_argument("--op", default="fprop", choices=["fprop", "fprop_int8", "dgrad", "wgrad", "graph", "peaks"],
                    help="fprop: the headline line; the others time the extensions on the same workload "
                         "(int8 output, data gradient, weight gradient, CUDA-graph replay vs eager calls), "
                         "or print the measured instruction-route rates (peaks)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------- ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (a host-side timing reduction only)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------- peaks, clocks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            return d, "measured"
        except (OSError, ValueError):
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _peak_value(peaks: dict, keys):
    for k in keys:
        v = peaks.get(k)
        if isinstance(v, (int, float)) and v > 0:
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "tflops", "gbs"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.gpu_id, self.period_ms = gpu_id, period_ms
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period_ms)], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        with open(self.tmp.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.tmp.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------- workloads on the device
ROTATE_MIN_BYTES = 16 << 20   # image+output sets at least this large rotate to keep L2 cold; smaller ones flush it
FLUSH_BYTES = 2 * L2_BYTES    # written between cold launches of the small workloads
HOST_AHEAD_CYCLES = 20_000_000  # GPU spin (~10 ms) before an event-timed loop: the host queues it meanwhile
IMAD_PER_SM_CLK = 64          # 32-bit integer multiply-adds per SM per clock (CUDA cores)


def workload_label(cfg) -> str:
    """The workload's name and every size that defines it (both arms print this)."""
    return (f"{cfg.name}: N={cfg.N} C={cfg.C} H={cfg.H} W={cfg.W} K={cfg.K} R={cfg.R} "
            f"S={cfg.S} stride={cfg.stride} pad={cfg.pre}/{cfg.post} dil={cfg.dilation} "
            f"mode={'conv' if cfg.mode else 'xcorr'} x={cfg.x_layout} w={cfg.w_layout} "
            f"y={cfg.y_layout} bias={cfg.bias} relu={cfg.relu}")


def rotating_sets(cfg) -> int:
    """Image/output sets to rotate over so that every call starts with a cold
    L2 (1: the set is small and the L2 is flushed instead)."""
    set_bytes = cfg.N * cfg.C * cfg.H * cfg.W + 4 * cfg.N * cfg.K * cfg.P * cfg.Q
    if set_bytes < ROTATE_MIN_BYTES:
        return 1
    return max(2, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)


class DeviceWorkload:
    """One workload resident on a device, called the way the benchmark times
    it, through the C ABI over ``nsets`` image/output sets: a step is one
    conv_fprop call (filter repack and convolution); pack() and conv() are
    its two halves as separate calls (conv_fprop_pack_filter,
    conv_fprop_prepacked), used to time the convolution alone."""

    def __init__(self, ic, cfg, dev, nsets: int = 1):
        import torch
        self.ic, self.cfg, self.dev, self.nsets = ic, cfg, dev, nsets
        self.x, self.w, self.b = synth.make_inputs(cfg)
        self.xf, self.xs = synth.place(self.x, cfg.x_layout)
        self.wf, self.ws = synth.place(self.w, cfg.w_layout)
        self.ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
        self.ysz = int(np.prod(cfg.y_dims))
        self.x_dev = [torch.from_numpy(self.xf).to(dev) for _ in range(nsets)]
        self.y_dev = [torch.empty(self.ysz, dtype=torch.int32, device=dev) for _ in range(nsets)]
        self.w_dev = torch.from_numpy(self.wf).to(dev)
        self.b_dev = torch.from_numpy(self.b).to(dev) if self.b is not None else None
        self.xd = ic.TensorDesc.make(ic.CONV_INT8, cfg.x_dims, self.xs, self.xf.size)
        self.wd = ic.TensorDesc.make(ic.CONV_INT8, cfg.w_dims, self.ws, self.wf.size)
        self.yd = ic.TensorDesc.make(ic.CONV_INT32, cfg.y_dims, self.ystr, self.ysz * 4)
        self.p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu)
        self.algo = ic.plan(self.xd, self.wd, self.yd, self.p)
        self.ws_bytes = ic.workspace_size(self.xd, self.wd, self.yd, self.p)
        self.work = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.kernels_per_step = ic.kernel_count(self.xd, self.wd, self.yd, self.p)
        self.bias_ptr = self.b_dev.data_ptr() if self.b_dev is not None else 0

    def pack(self, sh: int) -> None:
        st = self.ic.pack_filter_raw(self.xd, self.wd, self.w_dev.data_ptr(), self.yd, self.p, self.work.data_ptr(),
                                     self.ws_bytes, sh)
        if st:
            raise self.ic.ConvError(st, "pack filter")

    def conv(self, i: int, sh: int) -> None:
        s = i % self.nsets
        st = self.ic.conv_fprop_prepacked_raw(self.xd, self.x_dev[s].data_ptr(), self.wd, self.w_dev.data_ptr(),
                                              self.yd, self.y_dev[s].data_ptr(), self.bias_ptr, self.p,
                                              self.work.data_ptr(), self.ws_bytes, sh)
        if st:
            raise self.ic.ConvError(st, "conv")

    def step(self, i: int, sh: int) -> None:
        s = i % self.nsets
        st = self.ic.conv_fprop_raw(self.xd, self.x_dev[s].data_ptr(), self.wd, self.w_dev.data_ptr(), self.yd,
                                    self.y_dev[s].data_ptr(), self.bias_ptr, self.p, self.work.data_ptr(),
                                    self.ws_bytes, sh)
        if st:
            raise self.ic.ConvError(st, "conv_fprop")

    def output(self, i: int = 0) -> np.ndarray:
        """Logical [N,K,P,Q] int32 output of set i (after a synchronize)."""
        return synth.gather_logical(self.y_dev[i % self.nsets].cpu().numpy(), self.cfg.y_dims, self.ystr)


def roofline_of(cfg, algo_name: str, kernel_ms: float, peaks: dict, peak_src: str) -> dict:
    """Roofline of one convolution call: tensor floor (ops / bf16 peak) against
    the HBM floor (algorithmic bytes / copy bandwidth) for the tensor-core
    route, the CUDA cores' integer rate for the direct kernels."""
    bf16 = _peak_value(peaks, ("bf16_tflops", "bf16_dense_tflops"))
    bsrc = peak_src
    if bf16 is None:
        bf16, bsrc = FALLBACK_PEAKS["bf16_tflops"], "fallback"
    hbm = _peak_value(peaks, ("hbm_gbs",))
    hsrc = peak_src
    if hbm is None:
        hbm, hsrc = FALLBACK_PEAKS["hbm_gbs"], "fallback"
    alg_bytes = cfg.algorithmic_bytes()
    tensor_floor_ms = cfg.ops / (bf16 * 1e12) * 1e3
    hbm_floor_ms = alg_bytes / (hbm * 1e9) * 1e3
    r = {"kernel_ms": round(kernel_ms, 5), "algorithmic_bytes": alg_bytes,
         "tensor_floor_ms": round(tensor_floor_ms, 5), "hbm_floor_ms": round(hbm_floor_ms, 5)}
    if not algo_name.startswith("implicit_gemm"):
        alu = 152 * IMAD_PER_SM_CLK * 2 * 2.07e9 / 1e12
        ach = cfg.ops / (kernel_ms * 1e-3) / 1e12
        r.update({"bound": "alu", "achieved": round(ach, 6), "peak": round(alu, 2), "unit": "TOPS",
                  "frac": round(ach / alu, 6),
                  "peak_source": "152 SMs x 64 int32 multiply-adds/clk x 2 ops x 2.07 GHz (CUDA cores)"})
    elif hbm_floor_ms > tensor_floor_ms:
        gbs = alg_bytes / (kernel_ms * 1e-3) / 1e9
        r.update({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                  "frac": round(gbs / hbm, 4), "peak_source": f"{hsrc} HBM copy bandwidth",
                  "tensor_frac": round(cfg.ops / (kernel_ms * 1e-3) / 1e12 / bf16, 4)})
    else:
        ach = cfg.ops / (kernel_ms * 1e-3) / 1e12
        r.update({"bound": "tensor", "achieved": round(ach, 2), "peak": bf16, "unit": "TFLOP/s",
                  "frac": round(ach / bf16, 4),
                  "peak_source": f"{bsrc} bf16 dense burst (f16 operands run at the bf16 rate; sm_103a has "
                                 "no integer tcgen05 MMA)"})
    return r


def _median(v):
    return float(statistics.median(v)) if v else None


def time_workload(ic, cfg, dev, stream, flush, iters: int, warmup: int, peaks: dict, peak_src: str) -> dict:
    """Per-workload record: medians over ``iters`` event-timed launches of
    the step (repack + convolution) and of the convolution alone, each with a
    cold L2 (rotating sets, or a flush before each launch), and of the step
    with a warm L2 (one set, back to back)."""
    import torch
    nsets = rotating_sets(cfg)
    wl = DeviceWorkload(ic, cfg, dev, nsets)
    sh = stream.cuda_stream
    for i in range(warmup):
        wl.step(i, sh)
    torch.cuda.synchronize(dev)
    st = ic.device_status(sh)
    if st:
        raise ic.ConvError(st, f"{cfg.name} warm-up")

    def timed(fn, cold):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        for i in range(iters):
            if cold and nsets == 1:
                flush.zero_()
            evs[i][0].record(stream)
            fn(i + 1 if cold else 0)
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in evs]

    def looped(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(HOST_AHEAD_CYCLES)
        e0.record(stream)
        for i in range(iters):
            fn(i + 1)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / iters

    step_ms = timed(lambda i: wl.step(i, sh), True)
    # the convolution-only calls read the repacked filter (conv_fprop may
    # have converted the filter in its kernel, leaving the workspace unpacked)
    wl.pack(sh)
    conv_ms = timed(lambda i: wl.conv(i, sh), True)
    warm_ms = timed(lambda i: wl.step(i, sh), False)
    if nsets > 1:
        # launches back to back over the rotating sets (every one cold): the
        # average duration of a step and of a convolution call in a stream of
        # them, as in the headline's timed region
        step_avg, conv_avg = looped(lambda i: wl.step(i, sh)), looped(lambda i: wl.conv(i, sh))
    st = ic.device_status(sh)
    if st:
        raise ic.ConvError(st, f"{cfg.name} timed launches")
    algo = ic.ALGO_NAMES.get(wl.algo, str(wl.algo))
    if nsets > 1:
        ms, kms, how = step_avg, conv_avg, (f"average over {iters} back-to-back launches on rotating sets "
                                            f"(events at the ends)")
    else:
        ms, kms, how = _median(step_ms), _median(conv_ms), (f"median of {iters} launches, each after an L2 "
                                                            f"flush and timed with its own events")
    rec = {
        "workload": workload_label(cfg), "algo": algo, "ops": cfg.ops,
        "ms": round(ms, 5), "value": round(cfg.ops / (ms * 1e-3) / 1e12, 3), "unit": "TOPS",
        "kernel_ms": round(kms, 5), "kernel_share": round(kms / ms, 4), "timing": how,
        "kernel_ms_source": ("convolution-only calls (conv_fprop_prepacked, repacked filter); where the step's "
                             "one kernel converts the filter itself it is another kernel variant, and the "
                             "share can exceed 1"),
        "isolated_step_ms_median": round(_median(step_ms), 5),
        "isolated_kernel_ms_median": round(_median(conv_ms), 5),
        "warm_ms": round(_median(warm_ms), 5),
        "warm_value": round(cfg.ops / (_median(warm_ms) * 1e-3) / 1e12, 3),
        "launches_timed": iters, "kernels_per_step": wl.kernels_per_step,
        "l2": (f"cold: rotating {nsets} resident sets" if nsets > 1 else
               f"cold: {FLUSH_BYTES >> 20} MiB written before each launch") +
              "; warm: one set, launches back to back, median of their own events",
        "roofline": roofline_of(cfg, algo, kms, peaks, peak_src),
    }
    del wl
    torch.cuda.empty_cache()
    return rec


def measure_routes(ic, dev, sh) -> dict:
    """conv_measure_peak_rates over a 1 GiB scratch buffer: the dense rates of
    tcgen05 kind::f16 (the route taken), warp-level mma.sync s8 and f16, dp4a,
    and the copy bandwidth, with the SM clock seen."""
    import torch
    scratch = torch.empty((1 << 30) + 4096, dtype=torch.uint8, device=dev)
    r = ic.measure_peak_rates(scratch.data_ptr(), scratch.numel(), sh)
    del scratch
    torch.cuda.empty_cache()
    out = {k: round(v, 2) for k, v in r.items()}
    out["note"] = ("sm_103a has no integer tcgen05 MMA; the convolution takes tcgen05 kind::f16 (exact by "
                   "grouping), the fastest exact route measured here")
    return out


# ---------------------------------------------------------------------- oracle timing
def time_oracle_sample(cfg, seconds: float, x, w, b):
    """Time the CPU oracle on a random sample of output points sized to take
    about ``seconds``; returns (TOPS, threads, description, points)."""
    import oracle
    oracle.build()
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    rng = np.random.default_rng(1)

    def pts(n):
        return np.stack([rng.integers(0, d, n) for d in cfg.y_dims], axis=1)

    red = cfg.C * cfg.R * cfg.S
    probe = pts(max(64, int(2e7 // red)))
    t0 = time.perf_counter()
    oracle.conv_fprop_points(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, probe, cfg.pre, cfg.post, cfg.stride,
                             cfg.dilation, cfg.mode, b, cfg.relu)
    dt = max(time.perf_counter() - t0, 1e-6)
    n = max(256, int(len(probe) * seconds / dt))
    n = min(n, int(np.prod(cfg.y_dims)))
    sample = pts(n)
    t0 = time.perf_counter()
    oracle.conv_fprop_points(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, sample, cfg.pre, cfg.post, cfg.stride,
                             cfg.dilation, cfg.mode, b, cfg.relu)
    dt = time.perf_counter() - t0
    tops = 2.0 * n * red / dt / 1e12
    desc = (f"{n} randomly drawn output elements of the workload ({n * red * 2 / 1e9:.2f} G ops, "
            f"{100.0 * n / np.prod(cfg.y_dims):.3f}% of the outputs), seven-loop oracle, {dt:.1f} s")
    return tops, oracle.num_threads(), desc, n


def time_oracle_single_thread(names=("c1_tiny_nchw", "c2_s2_nhwc", "p4_shape")) -> dict:
    """The oracle on one core over the whole output of small workloads."""
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    out = {}
    try:
        oracle.set_num_threads(1)
        for name in names:
            cfg = synth.CONFIGS[name]
            x, w, b = synth.make_inputs(cfg)
            xf, xs = synth.place(x, cfg.x_layout)
            wf, ws = synth.place(w, cfg.w_layout)
            reps, dt = 0, 0.0
            t0 = time.perf_counter()
            while reps == 0 or (dt < 0.2 and reps < 10000):
                oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                                  cfg.dilation, cfg.mode, b, cfg.relu)
                reps += 1
                dt = time.perf_counter() - t0
            out[name] = {"ms": round(1e3 * dt / reps, 4), "tops": round(cfg.ops * reps / dt / 1e12, 8),
                         "ops": cfg.ops, "repeats": reps}
    finally:
        oracle.set_num_threads(threads)
    return out


# ---------------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    import int8_conv2d_fprop_gb300 as ic

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    cfg = synth.CONFIGS[args.workload]
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    peaks, peak_src = load_peaks()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(local)
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.15)

    # measured rates of the int8-capable instruction routes (rank 0)
    routes = None
    if rank == 0 and not args.no_peak_probe:
        routes = measure_routes(ic, dev, sh)

    # every workload of the specification, one record each (rank 0)
    per_workload = {}
    if rank == 0 and args.workloads:
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        for name in args.workloads.split(","):
            per_workload[name] = time_workload(ic, synth.CONFIGS[name], dev, stream, flush, args.launches,
                                               max(3, args.warmup if args.warmup < 20 else 20), peaks, peak_src)
        del flush
        torch.cuda.empty_cache()

    # the headline: exactly K steps of the workload, back to back
    nsets = max(2, rotating_sets(cfg))
    wl = DeviceWorkload(ic, cfg, dev, nsets)
    for i in range(args.warmup):
        wl.step(i, sh)
    torch.cuda.synchronize(dev)
    status = ic.device_status(sh)
    if status:
        raise ic.ConvError(status, "warm-up")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    torch.cuda._sleep(HOST_AHEAD_CYCLES)
    e0.record(stream)
    for i in range(args.steps):
        wl.step(args.warmup + i, sh)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    elapsed_ms = e0.elapsed_time(e1)
    status = ic.device_status(sh)
    if status:
        raise ic.ConvError(status, "timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    clocks = sampler.stop()
    if clocks:
        clocks["window"] = "whole GPU measurement (every workload's launches and the headline steps)"
    ms_per_step = elapsed_ms / args.steps
    value = world * cfg.ops / (ms_per_step * 1e-3) / 1e12
    algo_name = ic.ALGO_NAMES.get(wl.algo, str(wl.algo))
    gpu_launches = wl.kernels_per_step * args.steps

    # kernel time of the headline workload: the median of its own record (or
    # of a separate run of convolution-only launches when it has none)
    head = per_workload.get(cfg.name)
    if head is None:
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        head = time_workload(ic, cfg, dev, stream, flush, args.launches, 3, peaks, peak_src)
        del flush
    roofline = dict(head["roofline"])
    roofline["kernel"] = ("igemm_conv_kernel (+ igemm_split_reduce_kernel when the call cuts tiles)"
                          if algo_name.startswith("implicit_gemm") else algo_name)
    roofline["kernel_launches_timed"] = head["launches_timed"]
    roofline["kernel_ms_source"] = ("convolution-only calls (conv_fprop_prepacked) with a cold L2: " +
                                    head["timing"])
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        try:
            with open(TRAFFIC_FILE) as f:
                tr = json.load(f)
            src_sha = hashlib.sha256(open(DOMINANT_KERNEL_SRC, "rb").read()).hexdigest()
            entry = tr.get("workloads", {}).get(args.workload)
            if tr.get("kernel_src_sha256") == src_sha and entry:
                traffic = entry.get("dram_bytes_per_launch")
        except (OSError, ValueError):
            traffic = None
    roofline["traffic"] = traffic

    # end to end through the C ABI with host buffers (conv_fprop_host): every
    # step copies the image, filter and bias in from page-locked host memory
    # and the int32 output back, pipelined over the batch by the library
    e2e = None
    if args.e2e_steps > 0:
        xh = torch.from_numpy(wl.xf).pin_memory()
        wh = torch.from_numpy(wl.wf).pin_memory()
        bh = torch.from_numpy(wl.b).pin_memory() if wl.b is not None else None
        yh = torch.empty(wl.ysz, dtype=torch.int32).pin_memory()
        xd, wd, yd, p = wl.xd, wl.wd, wl.yd, wl.p
        del wl
        torch.cuda.empty_cache()
        hbytes = ic.host_buffer_size(xd, wd, yd, p)
        hbuf = torch.empty(hbytes, dtype=torch.uint8, device=dev)

        def e2e_step():
            st = ic.conv_fprop_host_raw(xd, xh.data_ptr(), wd, wh.data_ptr(), yd, yh.data_ptr(),
                                        bh.data_ptr() if bh is not None else 0, p, hbuf.data_ptr(), hbytes, sh)
            if st:
                raise ic.ConvError(st, "conv_fprop_host")

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        barrier(world)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev) / args.e2e_steps
        status = ic.device_status(sh)
        if status:
            raise ic.ConvError(status, "end-to-end")
        h2d = xh.numel() + wh.numel() + (bh.numel() * 4 if bh is not None else 0)
        e2e = {"value": round(world * cfg.ops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TOPS",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(yh.numel() * 4),
               "api": "conv_fprop_host (C ABI, page-locked host buffers, batch pipelined in chunks)"}
    else:
        del wl

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        x, w, b = synth.make_inputs(cfg)
        tops, threads, desc, _ = time_oracle_sample(cfg, args.cpu_seconds, x, w, b)
        cpu = {"value": round(tops, 6), "unit": "TOPS", "cores": threads, "kind": "oracle", "sample": desc,
               "single_thread": time_oracle_single_thread()}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8 x int8 -> int32 (exact, f16 tensor MMA)",
        "data": "synthetic (splitmix64 seeded int8 uniform[-128,127])",
        "config": {"workload": workload_label(cfg), "ops_per_step": cfg.ops, "algo": algo_name,
                   "l2": f"rotating {nsets} resident input/output sets (> 129 MB L2)",
                   "parallelism": f"replicas x{world}, no data-path collective"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "workloads": per_workload,
        "int8_routes": routes,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = synth.CONFIGS[args.workload]
    x, w, b = synth.make_inputs(cfg)
    import oracle
    oracle.build()
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    # size each step so that warm-up + timed steps take about 90 s in total
    per_step_s = max(0.05, min(2.0, 90.0 / max(1, args.steps + args.warmup)))
    _, threads, _, npts = time_oracle_sample(cfg, per_step_s, x, w, b)
    rng = np.random.default_rng(2)
    sample = np.stack([rng.integers(0, d, npts) for d in cfg.y_dims], axis=1)

    def step():
        oracle.conv_fprop_points(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, sample, cfg.pre, cfg.post, cfg.stride,
                                 cfg.dilation, cfg.mode, b, cfg.relu)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    red = cfg.C * cfg.R * cfg.S
    value = 2.0 * npts * red * args.steps / dt / 1e12
    desc = (f"each step: {npts} randomly drawn output elements of the workload "
            f"({2 * npts * red / 1e9:.3f} G ops) by the seven-loop CPU oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 x int8 -> int64 -> int32",
        "data": "synthetic (splitmix64 seeded int8 uniform[-128,127])",
        "config": {"workload": workload_label(cfg), "ops_per_step_sampled": int(2 * npts * red)},
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "kind": "oracle", "cores": threads,
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------- extensions


def run_extension(args):
    """One JSON line for an extension op on the workload, single GPU: the int8
    output epilogue, the data gradient, the weight gradient, or CUDA-graph
    replay of conv_fprop against eager calls.  Inputs resident, rotating sets
    larger than L2, CUDA events on the launching stream around every call."""
    import torch

    import int8_conv2d_fprop_gb300 as ic

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    cfg = synth.CONFIGS[args.workload]
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
    ysz = int(np.prod(cfg.y_dims))
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    peaks, peak_src = load_peaks()
    bf16 = _peak_value(peaks, ("bf16_tflops", "bf16_dense_tflops")) or FALLBACK_PEAKS["bf16_tflops"]
    if _peak_value(peaks, ("bf16_tflops", "bf16_dense_tflops")) is None:
        peak_src = "fallback"
    w_dev = torch.from_numpy(wf).to(dev)
    wd = ic.TensorDesc.make(ic.CONV_INT8, cfg.w_dims, ws, wf.size)
    xd = ic.TensorDesc.make(ic.CONV_INT8, cfg.x_dims, xs, xf.size)
    extra = {}

    if args.op in ("fprop_int8", "fprop", "graph"):
        int8 = args.op == "fprop_int8"
        esz = 1 if int8 else 4
        yd = ic.TensorDesc.make(ic.CONV_INT8 if int8 else ic.CONV_INT32, cfg.y_dims, ystr, ysz * esz)
        p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu,
                           out_shift=10 if int8 else None)
        set_bytes = xf.size + ysz * esz
        nsets = max(2, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1) if args.op != "graph" else 1
        a_sets = [torch.from_numpy(xf).to(dev) for _ in range(nsets)]
        o_sets = [torch.empty(ysz * esz, dtype=torch.uint8, device=dev) for _ in range(nsets)]
        b_dev = torch.from_numpy(b).to(dev) if b is not None else None
        wsb = ic.workspace_size(xd, wd, yd, p)
        work = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
        bias_ptr = b_dev.data_ptr() if b_dev is not None else 0

        def call(i, stream_handle=None):
            k = i % nsets
            st = ic.conv_fprop_raw(xd, a_sets[k].data_ptr(), wd, w_dev.data_ptr(), yd, o_sets[k].data_ptr(),
                                   bias_ptr, p, work.data_ptr(), wsb, stream_handle or sh)
            if st:
                raise ic.ConvError(st, "conv_fprop")

        ops = cfg.ops
        alg_bytes = xf.size + wf.size + ysz * esz + (4 * cfg.K if cfg.bias else 0)
        metric = ("INT8 conv fprop with int8 output TOPS (2NKPQCRS/s)" if int8 else
                  "INT8 conv fprop per-call latency, CUDA-graph replay vs eager (us)")
        bound, peak, unit = "tensor", bf16, "TFLOP/s"
    elif args.op == "dgrad":
        dy = synth.int8_uniform(cfg.seed, 3, cfg.y_dims)
        dyf, dys = synth.place(dy, cfg.y_layout)
        dyd = ic.TensorDesc.make(ic.CONV_INT8, cfg.y_dims, dys, dyf.size)
        dxs = synth.packed_strides(cfg.x_dims, cfg.x_layout)
        xsz = int(np.prod(cfg.x_dims))
        dxd = ic.TensorDesc.make(ic.CONV_INT32, cfg.x_dims, dxs, xsz * 4)
        p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode)
        set_bytes = dyf.size + xsz * 4
        nsets = max(2, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
        a_sets = [torch.from_numpy(dyf).to(dev) for _ in range(nsets)]
        o_sets = [torch.empty(xsz, dtype=torch.int32, device=dev) for _ in range(nsets)]
        wsb = ic.dgrad_workspace_size(dyd, wd, dxd, p)
        work = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
        L = ic.lib()

        def call(i):
            k = i % nsets
            st = L.conv_dgrad(ctypes.byref(dyd), a_sets[k].data_ptr(), ctypes.byref(wd), w_dev.data_ptr(),
                              ctypes.byref(dxd), o_sets[k].data_ptr(), ctypes.byref(p),
                              work.data_ptr() if wsb else None, wsb, sh)
            if st:
                raise ic.ConvError(st, "conv_dgrad")

        ops = cfg.ops
        alg_bytes = dyf.size + wf.size + xsz * 4
        metric = "INT8 conv dgrad TOPS (2NKPQCRS/s)"
        tensor = wsb > 0
        bound = "tensor" if tensor else "alu"
        peak = bf16 if tensor else 152 * IMAD_PER_SM_CLK * 2 * 2.07e9 / 1e12
        unit = "TFLOP/s" if tensor else "TOPS"
        extra["route"] = ("tensor cores (a forward convolution of dY per residue class of the stride)"
                          if tensor else "CUDA cores")
    else:  # wgrad
        dy = synth.int8_uniform(cfg.seed, 3, cfg.y_dims)
        dyf, dys = synth.place(dy, cfg.y_layout)
        dyd = ic.TensorDesc.make(ic.CONV_INT8, cfg.y_dims, dys, dyf.size)
        dws = synth.packed_strides(cfg.w_dims, cfg.w_layout)
        wsz = int(np.prod(cfg.w_dims))
        dwd = ic.TensorDesc.make(ic.CONV_INT32, cfg.w_dims, dws, wsz * 4)
        p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode)
        nsets = max(2, int(np.ceil(3 * L2_BYTES / (xf.size + dyf.size))) + 1)
        a_sets = [torch.from_numpy(xf).to(dev) for _ in range(nsets)]
        g_sets = [torch.from_numpy(dyf).to(dev) for _ in range(nsets)]
        out = torch.empty(wsz, dtype=torch.int32, device=dev)
        wsb = ic.wgrad_workspace_size(xd, dyd, dwd, p)
        work = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
        L = ic.lib()

        def call(i):
            k = i % nsets
            st = L.conv_wgrad(ctypes.byref(xd), a_sets[k].data_ptr(), ctypes.byref(dyd), g_sets[k].data_ptr(),
                              ctypes.byref(dwd), out.data_ptr(), ctypes.byref(p), work.data_ptr() if wsb else None,
                              wsb, sh)
            if st:
                raise ic.ConvError(st, "conv_wgrad")

        ops = cfg.ops
        alg_bytes = xf.size + dyf.size + wsz * 4
        metric = "INT8 conv wgrad TOPS (2NKPQCRS/s)"
        tensor = wsb > 0
        bound = "tensor" if tensor else "alu"
        unit = "TFLOP/s" if tensor else "TOPS"
        peak = bf16 if tensor else 152 * IMAD_PER_SM_CLK * 2 * 2.07e9 / 1e12
        n_batch, q_cols = cfg.y_dims[0], cfg.y_dims[3]
        fold = min(64 // n_batch, q_cols, 8) if n_batch <= 32 else 1
        extra["route"] = (("tensor cores (forward convolution of the image by dY, reduction split over the SMs"
                           + (f"; {fold} columns of dY folded into the channels per k-step" if fold > 1 else "")
                           + ")") if tensor else "CUDA cores")

    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize(dev)
    if ic.device_status(sh):
        raise RuntimeError("device status after warm-up")
    # the timed loop: events only at its ends (no per-call event records,
    # whose host cost would land in a host-bound call's time)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        call(args.warmup + i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    total_ms = e0.elapsed_time(e1)
    if ic.device_status(sh):
        raise RuntimeError("device status after the timed region")
    ms_per_step = total_ms / args.steps
    # device time of one call: a second pass with events around every call
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        evs[i][0].record(stream)
        call(args.warmup + args.steps + i)
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    call_ms = statistics.mean(a.elapsed_time(bb) for a, bb in evs)
    if ic.device_status(sh):
        raise RuntimeError("device status after the per-call pass")
    if args.op == "graph":
        # eager calls timed like the replays below: events only at the ends
        # of the loop, the C entry point called with arguments marshalled
        # once (what a caller that keeps its descriptors does)
        L = ic.lib()
        fn = L.conv_fprop
        xr, wr, yr, pr = ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd), ctypes.byref(p)
        xs_ptr = [t.data_ptr() for t in a_sets]
        ys_ptr = [t.data_ptr() for t in o_sets]
        wptr, wkptr = w_dev.data_ptr(), work.data_ptr()
        bptr = bias_ptr or None
        for i in range(args.warmup):
            fn(xr, xs_ptr[i % nsets], wr, wptr, yr, ys_ptr[i % nsets], bptr, pr, wkptr, wsb, sh)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for i in range(args.steps):
            k = i % nsets
            fn(xr, xs_ptr[k], wr, wptr, yr, ys_ptr[k], bptr, pr, wkptr, wsb, sh)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if ic.device_status(sh):
            raise RuntimeError("device status after the eager loop")
        eager_ms = e0.elapsed_time(e1) / args.steps
        # the same call captured once and replayed
        side = torch.cuda.Stream(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            call(0, side.cuda_stream)
        side.synchronize()
        # the call must be queued on the capturing stream to be recorded
        with torch.cuda.graph(graph, stream=side):
            call(0, side.cuda_stream)
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = g0.elapsed_time(g1) / args.steps
        line = {"metric": metric, "value": round(graph_ms * 1e3, 3), "unit": "us", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
                "eager_us": round(eager_ms * 1e3, 3), "graph_us": round(graph_ms * 1e3, 3),
                "eager_us_python_wrapper": round(ms_per_step * 1e3, 3),
                "gpu_call_us": round(call_ms * 1e3, 3),
                "config": {"workload": cfg.name, "l2": "one resident set (latency, not bandwidth)"},
                "data": "synthetic", "dtype": "int8 x int8 -> int32"}
        print(json.dumps(line), flush=True)
        return
    achieved = ops / (call_ms * 1e-3) / 1e12
    line = {
        "metric": metric, "value": round(ops / (ms_per_step * 1e-3) / 1e12, 3), "unit": "TOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "dtype": "int8 x int8 -> int32", "data": "synthetic (splitmix64 seeded int8 uniform[-128,127])",
        "config": {"workload": cfg.name, "op": args.op, "ops_per_step": ops,
                   "l2": f"rotating {nsets} resident sets (> 129 MB L2)", **extra},
        "roofline": {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": unit,
                     "frac": round(achieved / peak, 4), "peak_source": peak_src if bound == "tensor" else
                     "152 SMs x 64 int32 multiply-adds/clk x 2 ops x 2.07 GHz",
                     "call_ms": round(call_ms, 5), "algorithmic_bytes": int(alg_bytes)},
    }
    print(json.dumps(line), flush=True)


def run_peaks(args):
    import torch

    import int8_conv2d_fprop_gb300 as ic
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    r = measure_routes(ic, dev, torch.cuda.current_stream(dev).cuda_stream)
    peaks, src = load_peaks()
    line = {"metric": "measured dense rates of the int8-capable instruction routes", "routes": r,
            "driver_peaks": {k: peaks.get(k) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")},
            "driver_peaks_source": src}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "peaks":
        run_peaks(args)
    elif args.op != "fprop":
        run_extension(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
