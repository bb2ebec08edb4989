#!/usr/bin/env python
"""Benchmark of the ConvRot INT8 layer on GB300.

One step = the per-step hot path of a packed 20k-token training step of one
frozen ConvRot INT8 linear layer (x bf16 [20480, 4096], W [16384, 4096],
block 128): online rotation + per-row quantization of x, the fused int8 GEMM
with dequantization epilogue, rotation + quantization of dY along N, and the
int8 grad_x GEMM.  Weight quantization (with and without a LoRA merge), the
int8 backward weight preparation, the embedding-table quantization and the
quantized embedding lookup are load-time or separate kernels; each is timed
on its own workload and reported under "rows".

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ConvRot int8 linear TOPS & quantizer GB/s (1×GB300, % of roofline)"
WORKLOAD = ("train20k: packed 20k-token training step of one ConvRot INT8 linear layer, x bf16 [20480,4096] "
            "N(0,1) with 41 outlier channels x30, W bf16 [16384,4096] N(0,0.02), dY bf16 [20480,16384] N(0,1e-3), "
            "Hadamard block 128; per step: rotate+quantize x, widen W codes to a transient fp16 operand, int8 GEMM "
            "+ dequant -> y, rotate+quantize dY, widen the int8 backward weight, int8 grad_x GEMM -> dX")
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes (read + write) per launch of the GEMM (gemm_pair_kernel), from one-pass ncu
# captures (dram__bytes_read.sum + dram__bytes_write.sum) of
#   python -m int8_rotated_quantized_gb300.profile_case gemm_w16 --M 20480 --N 16384 --K 4096 --reps 3   (forward)
#   python -m int8_rotated_quantized_gb300.profile_case gemm_w16 --M 20480 --N 4096 --K 16384 --reps 3   (grad_x)
#   python -m int8_rotated_quantized_gb300.profile_case gemm_bf16 --M 20480 --N 4096 --K 16384 --reps 3  (bf16 grad_x)
# keyed by the hash of the kernel source they were taken on; reported as null
# once the kernel source differs (or where no capture was taken on it).
GEMM_TRAFFIC = {"source_sha256_16": "5d91db25bf865fff", "fwd": 1072621056 + 654961152, "bwd": 3197371136 + 162885120,
                "bf16_bwd": 3196183808 + 162829824}


def _gemm_source_current():
    import hashlib
    path = os.path.join(ROOT, "int8_rotated_quantized_gb300", "csrc", "gemm_tc.cu")
    try:
        with open(path, "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16] == GEMM_TRAFFIC["source_sha256_16"]
    except OSError:
        return False


def gemm_traffic_per_launch(key=None):
    """Measured DRAM bytes per launch (mean of the forward and grad_x shapes, or one key), or None."""
    if not _gemm_source_current():
        return None
    if key is not None:
        return GEMM_TRAFFIC[key]
    return (GEMM_TRAFFIC["fwd"] + GEMM_TRAFFIC["bwd"]) // 2


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ------------------------------------------------------------- multi-rank ----

def max_over_ranks(torch, dist, ms, device):
    """The job's time: the slowest rank's (all-reduce MAX; a no-op on one process)."""
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world, ops_per_step, steps, job_ms):
    """Whole-job TOPS: every rank runs its own batch (no data-path collective), so the
    work is world x steps x ops_per_step over the slowest rank's time."""
    return world * ops_per_step * steps / (job_ms * 1e-3) / 1e12


# ---------------------------------------------------------------- clocks ----

class NvmlSampler:
    """The SM clock and the clock-event reasons of one GPU, read through NVML
    (the driver's libnvidia-ml, read-only queries) every 2 ms on a background
    thread, so a timed region of tens of milliseconds still gets many samples."""

    NVML_CLOCK_SM = 1
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid, index: int):
        self.samples, self.reasons, self.max_mhz, self.lib = [], 0, None, None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            found = bool(uuid) and lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) == 0
            if not found and lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.reason_fn = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                              or getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None))
            self.lib, self.h = lib, h
        except (OSError, AttributeError):
            self.lib = None
            return
        self.stop_evt = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_evt.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(mhz)) == 0:
                self.samples.append(float(mhz.value))
            if self.reason_fn is not None and self.reason_fn(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= int(rs.value)
            time.sleep(0.002)

    def stop(self):
        if self.lib is None:
            return None
        self.stop_evt.set()
        self.thread.join(timeout=5)
        names = sorted(n for bit, n in self.REASON_BITS.items() if self.reasons & bit)
        return {"samples": list(self.samples), "max_mhz": self.max_mhz, "reasons": names}


def gpu_uuid(torch, dev):
    u = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    return str(u) if u is not None else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms in the background,
    plus the in-process NVML sampler for short regions."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, uuid=None):
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        self.proc = None
        self.nvml = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", ("GPU-" + uuid) if uuid else str(gpu_index),
                                          f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def start_fine(self, gpu_index: int, uuid=None):
        """Begin the 2 ms NVML sampling (call right before the timed region)."""
        self.nvml = NvmlSampler(uuid, gpu_index)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.strip().split(",") for ln in self.file.read().splitlines() if ln.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for name, val in zip(names, r[5:9]):
                    if val.strip().lower() in ("active", "0x1", "1"):
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        source = "nvidia-smi every 100 ms"
        fine = self.nvml.stop() if self.nvml is not None else None
        if fine and fine["samples"]:
            # the median comes from the timed region alone; reasons from both samplers
            sm = fine["samples"]
            mx = max(mx, fine["max_mhz"] or 0.0)
            reasons |= set(fine["reasons"])
            source = "NVML every 2 ms during the timed region (reasons also from nvidia-smi every 100 ms)"
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "source": source}


# ------------------------------------------------------------ our kernels ----

def run_gpu(args):
    import torch
    import torch.distributed as dist

    import int8_rotated_quantized_gb300 as cr
    import synth
    import synth.gpu as sg
    from int8_rotated_quantized_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    cr.lib()
    pk = peaks()

    wl = synth.WORKLOADS["train20k"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    # weak scaling: every rank owns its own 20480-token batch (rows row0 .. row0+M of one tall batch)
    row0 = rank * M
    x = sg.activations_bf16(0, M, K, wl["x_outliers"], wl["x_factor"], dev, row0=row0)
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], dev)
    dY = sg.normal_bf16(0, synth.STREAM_DY, M, N, wl["dy_sigma"], dev, row0=row0)
    stream = torch.cuda.current_stream()

    # load-time work (not in the step): quantize W, prepare the int8 backward weight
    Wq, sw = cr.convrot_quantize_weight(W, b)
    WtQ, swt = cr.convrot_prepare_bwd_weight(Wq, sw, b)
    xq = torch.empty((M, K), dtype=torch.float16, device=dev)
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    dyq = torch.empty((M, N), dtype=torch.float16, device=dev)
    sdy = torch.empty((M,), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert cr.convrot_get_error() == cr.OK

    # transient fp16 copies of the weight codes (the int8 weights stay int8 at rest)
    w16 = torch.empty((N, K), dtype=torch.float16, device=dev)
    wt16 = torch.empty((K, N), dtype=torch.float16, device=dev)

    def step(ev=None):
        def mark(i):
            if ev:
                ev[i].record(stream)
        mark(0)
        cr.convrot_quantize_activation(x, b, xq, sx)
        mark(1)
        cr.convrot_widen_codes(Wq, w16)
        mark(2)
        cr.convrot_gemm_dequant_w16(xq, sx, w16, sw, None, y)
        mark(3)
        cr.convrot_quantize_activation(dY, b, dyq, sdy)
        mark(4)
        cr.convrot_widen_codes(WtQ, wt16)
        mark(5)
        cr.convrot_gemm_dequant_w16(dyq, sdy, wt16, swt, None, dX)
        mark(6)

    launches_per_step = 6
    uuid = gpu_uuid(torch, dev)
    sampler = ClockSampler(local, uuid) if rank == 0 else None
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert cr.convrot_get_error() == cr.OK

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    if sampler is not None:
        sampler.start_fine(local, uuid)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()  # L2 flush between steps, outside the events
        step(evs[i])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop() if sampler else None

    step_ms = [e[0].elapsed_time(e[6]) for e in evs]
    k1x = [e[0].elapsed_time(e[1]) for e in evs]
    wf = [e[1].elapsed_time(e[2]) for e in evs]
    gf = [e[2].elapsed_time(e[3]) for e in evs]
    k1d = [e[3].elapsed_time(e[4]) for e in evs]
    wb = [e[4].elapsed_time(e[5]) for e in evs]
    gb = [e[5].elapsed_time(e[6]) for e in evs]
    total_ms = max_over_ranks(torch, dist, sum(step_ms), dev)
    assert cr.convrot_get_error() == cr.OK

    ops_step = 2.0 * 2.0 * M * N * K           # fwd + grad_x GEMMs
    value = weak_scaling_value(world, ops_step, args.steps, total_ms)
    gemm_ms = statistics.mean(gf + gb)
    gemm_tflops = 2.0 * M * N * K / (gemm_ms * 1e-3) / 1e12

    result = None
    if rank == 0:
        int8_peak = measure_int8_mma_peak(cr, torch, dev)
        rows = measure_rows(cr, synth, sg, torch, dev, flush, pk, int8_peak) if not args.no_rows else {}
        # the method's own output is 1-byte codes (+ fp32 scales): those are the algorithmic bytes;
        # the fp16 container the GEMM reads is reported beside them
        rows["a3_x_rotate_quant"] = _hbm_row(M * K * 2 + M * K + M * 4, statistics.median(k1x), pk,
                                             "train20k x [20480,4096] bf16 -> codes (held as fp16) + fp32 scales",
                                             container_bytes=M * K * 2 + M * K * 2 + M * 4)
        rows["a6_dy_rotate_quant"] = _hbm_row(M * N * 2 + M * N + M * 4, statistics.median(k1d), pk,
                                              "train20k dY [20480,16384] bf16 -> codes (held as fp16) + fp32 scales",
                                              container_bytes=M * N * 2 + M * N * 2 + M * 4)
        rows["overhead_widen_weight_codes"] = _overhead_row(
            3 * N * K, statistics.median(wf + wb), 2, statistics.median(step_ms),
            "train20k: int8 weight codes [16384,4096] -> transient fp16 operand, once before each GEMM (forward "
            "and grad_x); work the method does not have, the price of the fp16 tensor-core route")
        rows["a4a5_fwd_gemm"] = _tc_row(2.0 * M * N * K, statistics.median(gf), pk, "train20k 20480x16384x4096",
                                        int8_peak)
        rows["a6_bwd_gemm"] = _tc_row(2.0 * M * N * K, statistics.median(gb), pk, "train20k 20480x4096x16384",
                                      int8_peak)
        e2e = measure_e2e(cr, torch, dev, x, dY, Wq, sw, WtQ, swt, b, ops_step, steps=max(4, args.steps))
        cpu = None
        if world == 1 and not args.no_cpu:
            cpu = cpu_baseline(args.cpu_rows, M, K, N, b, wl)
        result = {
            "metric": METRIC,
            "value": round(value, 3),
            "unit": "TOPS",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "s8",
            "data": "synthetic (seeded splitmix64 + Box-Muller, generated on the device)",
            "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "block": b,
                       "tokens_per_gpu": M, "l2": "flushed between steps (256 MiB write, outside the events)",
                       "parallelism": f"replicas x{world} (rows sharded, no collective)"},
            "roofline": {
                "kernel": "gemm_pair_kernel (CTA pairs, 2-SM MMA), widened-weight mode (fwd and grad_x launches)",
                "bound": "tensor",
                "achieved": round(gemm_tflops, 1),
                "peak": pk["bf16"],
                "unit": "TFLOP/s",
                "frac": round(gemm_tflops / pk["bf16"], 4),
                "peak_note": f"{pk['source']} dense bf16 burst (the kind::f16 MMA that carries the int8 codes runs at the "
                             "bf16/fp16 rate; tcgen05 kind::i8 does not exist on sm_103a)",
                "int8_peak": int8_peak["TOPS"],
                "frac_of_int8_peak": round(gemm_tflops / int8_peak["TOPS"], 3),
                "int8_peak_note": "measured in this run: dense int8 through the only int8 MMA of sm_103a, the legacy "
                                  "warp-level mma.sync m16n8k32 s8 (convrot_probe_mma_s8_rate, "
                                  f"{int8_peak['ms']} ms for {int8_peak['ops']:.3e} ops, 4 CTAs x 8 warps per SM)",
                "traffic": gemm_traffic_per_launch(),
                "traffic_note": "mean DRAM bytes per launch over the forward and grad_x shapes (ncu, one pass); "
                                "algorithmic bytes per launch 973225984 for both (fp16 activation and weight "
                                "codes, bf16 output, fp32 scales)",
            },
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "wall_s_timed_region": round(t_wall, 4),
            "rows": rows,
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return result


def fp32_fma_peak(torch, dev):
    """fp32 fused multiply-adds per second: 128 lanes per SM per clock at the maximum SM clock."""
    props = torch.cuda.get_device_properties(dev)
    mhz = 2070.0
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=clocks.max.sm", "--format=csv,noheader,nounits", "-i",
                              str(dev.index or 0)], capture_output=True, text=True, timeout=10).stdout.strip()
        mhz = float(out.splitlines()[0])
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        pass
    return props.multi_processor_count * 128 * mhz * 1e6


def _hbm_row(nbytes, ms, pk, what, container_bytes=None):
    """An HBM-bound row: GB/s and frac on the algorithmic bytes (the compulsory reads and
    writes of the method's own data: bf16 in, 1-byte codes, fp32 scales); where the kernel
    writes a wider container (fp16-held codes), its bytes and rate are reported beside."""
    gbs = nbytes / (ms * 1e-3) / 1e9
    row = {"what": what, "ms": round(ms, 4), "algorithmic_bytes": int(nbytes), "GB/s": round(gbs, 1),
           "peak_GB/s": pk["hbm"], "frac": round(gbs / pk["hbm"], 4)}
    if container_bytes is not None:
        cgbs = container_bytes / (ms * 1e-3) / 1e9
        row.update({"container_bytes": int(container_bytes), "container_GB/s": round(cgbs, 1),
                    "container_frac": round(cgbs / pk["hbm"], 4)})
    return row


def _overhead_row(nbytes, ms, launches, step_ms, what):
    """Work the method does not have (no roofline achievement): its time and share of the step."""
    return {"what": what, "overhead": True, "ms_per_launch": round(ms, 4), "launches_per_step": launches,
            "ms_per_step": round(ms * launches, 4), "share_of_step": round(ms * launches / step_ms, 4),
            "bytes_moved_per_launch": int(nbytes), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}


def _tc_row(ops, ms, pk, what, int8_peak=None):
    tops = ops / (ms * 1e-3) / 1e12
    row = {"what": what, "ms": round(ms, 4), "ops": ops, "TOPS": round(tops, 1), "peak_TFLOP/s": pk["bf16"],
           "frac": round(tops / pk["bf16"], 4)}
    if int8_peak is not None:
        row.update({"int8_peak_TOPS": int8_peak["TOPS"], "frac_of_int8_peak": round(tops / int8_peak["TOPS"], 3)})
    return row


def measure_int8_mma_peak(cr, torch, dev, reps=5):
    """Dense int8 rate of the legacy warp-level MMA (the only int8 MMA on sm_103a), timed
    with CUDA events around the library's probe kernel; the median of `reps` launches."""
    sink = torch.empty(1 << 16, dtype=torch.int32, device=dev)
    ops = ctypes.c_double()
    stream = torch.cuda.current_stream()

    def launch(iters):
        rc = cr.lib().convrot_probe_mma_s8_rate(iters, cr._ptr(sink), sink.numel() * 4, ctypes.byref(ops),
                                                cr._stream(None))
        assert rc == cr.OK
    launch(64)
    torch.cuda.synchronize()
    iters, ms = 4096, []
    for _ in range(reps + 1):
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        launch(iters)
        z.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(z))
    t = statistics.median(ms[1:])
    return {"TOPS": round(ops.value / (t * 1e-3) / 1e12, 1), "ms": round(t, 3), "ops": ops.value}


def _time(torch, fn, flush, reps, pre=None):
    """Median device time (ms) of fn() over reps, each after an L2 flush."""
    stream = torch.cuda.current_stream()
    out = []
    for i in range(reps + 2):
        flush.zero_()
        if pre:
            pre(i)
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(i)
        z.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            out.append(a.elapsed_time(z))
    return statistics.median(out)


def measure_rows(cr, synth, sg, torch, dev, flush, pk, int8_peak=None):
    rows = {}
    reps = 10
    # the single 1024^2-image forward: x [4096,4096] (4096 image tokens), W [4096,4096]
    wl2 = synth.WORKLOADS["img1024"]
    M2, K2, N2, b2 = wl2["M"], wl2["K"], wl2["N"], wl2["block"]
    x2 = sg.activations_bf16(0, M2, K2, wl2["x_outliers"], wl2["x_factor"], dev)
    W2 = sg.normal_bf16(0, synth.STREAM_W, N2, K2, wl2["w_sigma"], dev)
    xq2 = torch.empty((M2, K2), dtype=torch.float16, device=dev)
    sx2 = torch.empty((M2,), dtype=torch.float32, device=dev)
    Wq2 = torch.empty((N2, K2), dtype=torch.int8, device=dev)
    sw2 = torch.empty((N2,), dtype=torch.float32, device=dev)
    ms = _time(torch, lambda i: cr.convrot_quantize_activation(x2, b2, xq2, sx2), flush, reps)
    rows["c2_a3_x_rotate_quant"] = _hbm_row(M2 * K2 * 3 + M2 * 4, ms, pk,
                                            "img1024 x [4096,4096] bf16 -> codes (held as fp16) + fp32 scales",
                                            container_bytes=M2 * K2 * 4 + M2 * 4)
    ms = _time(torch, lambda i: cr.convrot_quantize_weight(W2, b2, Wq=Wq2, scale_w=sw2), flush, reps)
    rows["c2_a2_weight_rotate_quant"] = _hbm_row(N2 * K2 * 3 + N2 * 4, ms, pk, "img1024 W [4096,4096] bf16 -> int8")
    w16 = cr.convrot_widen_codes(Wq2)
    y2 = torch.empty((M2, N2), dtype=torch.bfloat16, device=dev)
    ms = _time(torch, lambda i: cr.convrot_gemm_dequant_w16(xq2, sx2, w16, sw2, None, y2), flush, reps)
    tiles = -(-M2 // 256) * -(-N2 // 256)
    rows["c2_a4a5_gemm"] = _tc_row(2.0 * M2 * N2 * K2, ms, pk,
                                   f"img1024 4096x4096x4096 GEMM + dequant (widened-weight mode; {tiles} tiles of "
                                   "256 tokens x 256 weight rows on CTA pairs, one per two SMs)", int8_peak)
    ws2 = torch.empty(cr.convrot_linear_workspace_bytes(M2, K2, N2), dtype=torch.uint8, device=dev)
    ms = _time(torch, lambda i: cr.convrot_linear_fwd(x2, Wq2, sw2, b2, y=y2, workspace=ws2), flush, reps)
    rows["c2_fwd_call"] = _tc_row(2.0 * M2 * N2 * K2, ms, pk,
                                  "img1024 whole forward call (rotate+quantize x, widen W codes, GEMM + dequant)",
                                  int8_peak)
    ms = _time(torch, lambda i: cr.convrot_linear_fwd_noalloc(x2, Wq2, sw2, b2, y=y2), flush, reps)
    rows["c2_fwd_noalloc_call"] = _tc_row(2.0 * M2 * N2 * K2, ms, pk,
                                          "img1024 forward without a workspace (library-owned code array; the GEMM "
                                          "widens the int8 weight codes in its loop)", int8_peak)
    del x2, W2, xq2, sx2, Wq2, sw2, w16, y2, ws2
    # a2: weight rotate + quantize, the 20k-token workload's weight
    wl = synth.WORKLOADS["train20k"]
    N, K, b = wl["N"], wl["K"], wl["block"]
    W = sg.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"], dev)
    Wq = torch.empty((N, K), dtype=torch.int8, device=dev)
    sw = torch.empty((N,), dtype=torch.float32, device=dev)
    ms = _time(torch, lambda i: cr.convrot_quantize_weight(W, b, Wq=Wq, scale_w=sw), flush, reps)
    rows["a2_weight_rotate_quant"] = _hbm_row(N * K * 2 + N * K + N * 4, ms, pk, "train20k W [16384,4096] bf16 -> int8")
    # a6 prep (one-off): int8 backward weight
    WtQ = torch.empty((K, N), dtype=torch.int8, device=dev)
    swt = torch.empty((K,), dtype=torch.float32, device=dev)
    ws = torch.empty(cr.convrot_bwd_weight_workspace_bytes(N, K), dtype=torch.uint8, device=dev)
    ms = _time(torch, lambda i: cr.convrot_prepare_bwd_weight(Wq, sw, b, WtQ, swt, ws), flush, 3)
    rows["a6_prep_bwd_weight"] = _hbm_row(N * K + N * 4 + K * N + K * 4, ms, pk,
                                          "train20k Wq [16384,4096] -> WtQ [4096,16384] (one-off, via a double-float workspace)")
    del ws
    # the bf16 backward mode (transient dequantization + bf16 tcgen05 GEMM), on the 20k-token shapes
    M = wl["M"]
    weff_t = torch.empty((K, N), dtype=torch.bfloat16, device=dev)
    ms = _time(torch, lambda i: cr.convrot_dequant_weight_t(Wq, sw, b, weff_t), flush, reps)
    rows["n1_bf16_bwd_dequant"] = _hbm_row(N * K + N * 4 + K * N * 2, ms, pk,
                                           "train20k Wq [16384,4096] -> W_eff^T bf16 [4096,16384] (per backward)")
    dY = sg.normal_bf16(0, synth.STREAM_DY, M, N, wl["dy_sigma"], dev)
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    ms = _time(torch, lambda i: cr.convrot_gemm_bf16(dY, weff_t, dX), flush, 5)
    rows["n1_bf16_bwd_gemm"] = _tc_row(2.0 * M * N * K, ms, pk, "train20k dY [20480,16384] . W_eff -> dX bf16 [20480,4096]")
    rows["n1_bf16_bwd_gemm"].update({"traffic": gemm_traffic_per_launch("bf16_bwd"),
                                     "algorithmic_bytes": M * N * 2 + K * N * 2 + M * K * 2})
    # the second reading of the int8 backward (no prepared weight copy), and the accuracy of the
    # two int8 readings against the bf16 mode on this workload
    ws3 = torch.empty(cr.convrot_bwd_x_r2_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    dX3 = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    ms = _time(torch, lambda i: cr.convrot_linear_bwd_x_r2(dY, Wq, sw, b, dX3, ws3), flush, 5)
    rows["n3_int8_bwd_second_reading"] = _tc_row(2.0 * M * N * K, ms, pk,
                                                 "train20k dY [20480,16384] -> dX [20480,4096], scale-folded unrotated "
                                                 "codes, Wq as stored, rotation of the product (whole call)")
    dX1 = cr.convrot_linear_bwd_x(dY, WtQ, swt, b)
    cr.convrot_gemm_bf16(dY, cr.convrot_dequant_weight_t(Wq, sw, b), dX)

    def rel(a):
        return round(float(torch.linalg.vector_norm((a.float() - dX.float())) / torch.linalg.vector_norm(dX.float())), 5)
    rows["n3_int8_bwd_second_reading"].update({"rel_fro_vs_bf16_mode": rel(dX3),
                                               "first_reading_rel_fro_vs_bf16_mode": rel(dX1)})
    del W, Wq, weff_t, dY, dX, dX1, dX3, ws3, WtQ
    # a1 + a2: LoRA merge fused into the weight quantizer, the qkv weight
    wl3 = synth.WORKLOADS["qkv_lora"]
    N3, K3, r = wl3["N"], wl3["K"], wl3["lora_rank"]
    W3 = sg.normal_bf16(0, synth.STREAM_W, N3, K3, wl3["w_sigma"], dev)
    A, B = sg.lora_pair(0, N3, K3, r, wl3["lora_sigma"], dev)
    Wq3 = torch.empty((N3, K3), dtype=torch.int8, device=dev)
    sw3 = torch.empty((N3,), dtype=torch.float32, device=dev)
    ms = _time(torch, lambda i: cr.convrot_quantize_weight(W3, b, A, B, wl3["lora_alpha"], wl3["lora_scale"], Wq3,
                                                           sw3), flush, reps)
    rows["a1a2_lora_merge_quant"] = _hbm_row(N3 * K3 * 2 + N3 * K3 + N3 * 4 + r * K3 * 4 + N3 * r * 4, ms, pk,
                                             "qkv W [12288,4096] + LoRA r16 -> int8")
    # the merge is r + 1 fp32 fused multiply-adds per element in a fixed order: its ALU roofline
    fma = N3 * K3 * (r + 1)
    fma_peak = fp32_fma_peak(torch, dev)
    rows["a1a2_lora_merge_quant"].update({"fma_per_s_T": round(fma / (ms * 1e-3) / 1e12, 2),
                                          "fma_peak_T": round(fma_peak / 1e12, 2),
                                          "fma_frac": round(fma / (ms * 1e-3) / fma_peak, 4)})
    # the same adapter as an unmerged bypass in the forward (x [4096,4096] of the qkv workload)
    M3 = wl3["M"]
    x3 = sg.activations_bf16(0, M3, K3, wl3["x_outliers"], wl3["x_factor"], dev)
    Wq3p, sw3p = cr.convrot_quantize_weight(W3, b)
    y3 = torch.empty((M3, N3), dtype=torch.bfloat16, device=dev)
    wsl = torch.empty(cr.convrot_linear_lora_workspace_bytes(M3, K3, N3), dtype=torch.uint8, device=dev)
    wsp = torch.empty(cr.convrot_linear_workspace_bytes(M3, K3, N3), dtype=torch.uint8, device=dev)
    ms_l = _time(torch, lambda i: cr.convrot_linear_fwd_lora(x3, Wq3p, sw3p, b, A, B, wl3["lora_alpha"],
                                                             wl3["lora_scale"], y=y3, workspace=wsl), flush, reps)
    ms_p = _time(torch, lambda i: cr.convrot_linear_fwd(x3, Wq3p, sw3p, b, y=y3, workspace=wsp), flush, reps)
    rows["n2_lora_bypass_fwd"] = _tc_row(2.0 * M3 * N3 * K3, ms_l, pk,
                                         "qkv x [4096,4096] . W [12288,4096] + LoRA r16 bypass, whole forward call")
    rows["n2_lora_bypass_fwd"].update({"plain_fwd_ms": round(ms_p, 4),
                                       "bypass_overhead_frac": round(ms_l / ms_p - 1.0, 4)})
    rows["c3_fwd_call"] = _tc_row(2.0 * M3 * N3 * K3, ms_p, pk,
                                  "qkv x [4096,4096] . W [12288,4096] (LoRA merged at load), whole forward call "
                                  "(rotate+quantize x, widen W codes, GEMM + dequant)", int8_peak)
    xq3, sx3 = cr.convrot_quantize_activation(x3, b)
    w16_3 = cr.convrot_widen_codes(Wq3)
    ms = _time(torch, lambda i: cr.convrot_gemm_dequant_w16(xq3, sx3, w16_3, sw3, None, y3), flush, reps)
    rows["c3_a4a5_gemm"] = _tc_row(2.0 * M3 * N3 * K3, ms, pk,
                                   "qkv 4096x12288x4096 GEMM + dequant (widened-weight mode, merged weight)", int8_peak)
    del W3, Wq3, A, B, x3, Wq3p, sw3p, y3, wsl, wsp, xq3, sx3, w16_3
    # a7: embedding table quantization (row-chunked: 8 slabs of 31000 rows)
    wl5 = synth.WORKLOADS["embed"]
    V, D = wl5["V"], wl5["D"]
    T = sg.normal_bf16(0, synth.STREAM_TABLE, V, D, wl5["table_sigma"], dev)
    Eq = torch.empty((V, D), dtype=torch.int8, device=dev)
    se = torch.empty((V,), dtype=torch.float32, device=dev)
    slab = 31000

    def quant_table(i):
        for r0 in range(0, V, slab):
            r1 = min(V, r0 + slab)
            cr.convrot_quantize_weight(T[r0:r1], b, Wq=Eq[r0:r1], scale_w=se[r0:r1])

    ms = _time(torch, quant_table, flush, 5)
    rows["a7_table_rotate_quant"] = _hbm_row(V * D * 2 + V * D + V * 4, ms, pk,
                                             "embed table [248000,4096] bf16 -> int8, 8 row slabs")
    del T
    # a8: lookup of 8192 ids, rotating over 8 id sets
    n_ids = wl5["n_ids"]
    id_sets = [sg.token_ids(0, n_ids, V, dev, set_index=s) for s in range(wl5["id_sets"])]
    out = torch.empty((n_ids, D), dtype=torch.bfloat16, device=dev)
    ms = _time(torch, lambda i: cr.convrot_embedding_lookup(id_sets[i % len(id_sets)], Eq, se, b, out), flush, 16)
    rows["a8_embedding_lookup"] = _hbm_row(n_ids * 8 + n_ids * D + n_ids * 4 + n_ids * D * 2, ms, pk,
                                           "embed 8192 ids -> bf16 [8192,4096]")
    assert cr.convrot_get_error() == cr.OK
    del Eq, se, out, id_sets
    add_same_size_copy(torch, dev, flush, rows)
    return rows


def add_same_size_copy(torch, dev, flush, rows):
    """Context for the memory-bound rows: a device-to-device copy (torch) that moves the
    same number of bytes, timed the same way.  Launch and ramp cost a visible share of
    kernels of a few tens of microseconds, which the large-copy peak does not show."""
    for row in rows.values():
        nbytes = row.get("algorithmic_bytes")
        if not nbytes or "GB/s" not in row:
            continue
        half = max(int(nbytes // 2) // 256 * 256, 256)
        a = torch.empty(half, dtype=torch.uint8, device=dev)
        c = torch.empty_like(a)
        ms = _time(torch, lambda i: c.copy_(a), flush, 9)
        copy_gbs = 2 * half / (ms * 1e-3) / 1e9
        row["same_size_copy_GB/s"] = round(copy_gbs, 1)
        row["frac_of_same_size_copy"] = round(row["GB/s"] / copy_gbs, 4)
        del a, c


def measure_e2e(cr, torch, dev, x, dY, Wq, sw, WtQ, swt, b, ops_step, steps=20):
    """The step through the public calls with host buffers: every step copies its
    x and dY from pinned host memory to the device, runs the forward and grad_x
    calls, and copies y and dX back to pinned host memory, all inside the timed
    region.  The copies run on their own streams (host-to-device, device-to-host)
    with double-buffered device tensors, so a step's transfers overlap the
    neighbouring steps' kernels; events order every reuse of a buffer."""
    M, K = x.shape
    N = dY.shape[1]
    xh = x.cpu().pin_memory()
    dyh = dY.cpu().pin_memory()
    yh = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dxh = [torch.empty((M, K), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    dyd = [torch.empty_like(dY) for _ in range(2)]
    yd = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    dxd = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws = torch.empty(max(cr.convrot_linear_workspace_bytes(M, K, N), cr.convrot_linear_workspace_bytes(M, N, K)),
                     dtype=torch.uint8, device=dev)
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    x_in, dy_in, comp_done, y_ready, dx_ready, out_done = ([ev() for _ in range(2)] for _ in range(6))
    used = [False, False]

    def one(i):
        j = i % 2
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(comp_done[j])           # step i-2 no longer reads xd[j], dyd[j]
            xd[j].copy_(xh, non_blocking=True)
            x_in[j].record(s_in)
            dyd[j].copy_(dyh, non_blocking=True)
            dy_in[j].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(x_in[j])
            if used[j]:
                s_comp.wait_event(out_done[j])          # step i-2's results have left yd[j], dxd[j]
            cr.convrot_linear_fwd(xd[j], Wq, sw, b, y=yd[j], workspace=ws, stream=s_comp)
            y_ready[j].record(s_comp)
            s_comp.wait_event(dy_in[j])
            cr.convrot_linear_bwd_x(dyd[j], WtQ, swt, b, dX=dxd[j], workspace=ws, stream=s_comp)
            dx_ready[j].record(s_comp)
            comp_done[j].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(y_ready[j])
            yh[j].copy_(yd[j], non_blocking=True)
            s_out.wait_event(dx_ready[j])
            dxh[j].copy_(dxd[j], non_blocking=True)
            out_done[j].record(s_out)
        used[j] = True

    one(0)
    one(1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    return {"value": round(ops_step / dt / 1e12, 3), "unit": "TOPS", "ms_per_step": round(dt * 1e3, 3),
            "h2d_bytes_per_step": int(x.numel() * 2 + dY.numel() * 2),
            "d2h_bytes_per_step": int(M * N * 2 + M * K * 2),
            "steps": steps,
            "schedule": "3 streams (host-to-device copies, kernels, device-to-host copies), double-buffered; "
                        "wall clock over the steps, synchronised on both sides"}


# ---------------------------------------------------------------- oracle ----

def _oracle_setup(M, K, N, b, wl, rows):
    import numpy as np  # noqa: F401

    import oracle
    import synth
    oracle.build()
    W = synth.normal_bf16(0, synth.STREAM_W, N, K, wl["w_sigma"])
    wq, sw = oracle.quantize_weight(W, b)
    wtq, swt = oracle.prepare_bwd_weight(wq, sw, b)
    x = synth.activations_bf16(0, rows, K, wl["x_outliers"], wl["x_factor"])
    dy = synth.normal_bf16(0, synth.STREAM_DY, rows, N, wl["dy_sigma"])
    return oracle, (wq, sw, wtq, swt, x, dy)


def _oracle_step(oracle, data, b):
    wq, sw, wtq, swt, x, dy = data
    oracle.linear_fwd(x, wq, sw, b)
    oracle.linear_bwd_x(dy, wtq, swt, b)


def cpu_baseline(rows, M, K, N, b, wl):
    oracle, data = _oracle_setup(M, K, N, b, wl, rows)
    t0 = time.perf_counter()
    _oracle_step(oracle, data, b)
    dt = time.perf_counter() - t0
    return {"value": round(2.0 * 2.0 * rows * N * K / dt / 1e12, 6), "unit": "TOPS", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{rows} of the {M} token rows of one step (fwd + grad_x), weights prepared outside the timing; "
                      f"{dt:.2f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import synth
    wl = synth.WORKLOADS["train20k"]
    M, K, N, b = wl["M"], wl["K"], wl["N"], wl["block"]
    oracle, data = _oracle_setup(M, K, N, b, wl, args.ref_rows)
    for _ in range(args.warmup):
        _oracle_step(oracle, data, b)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(oracle, data, b)
    dt = time.perf_counter() - t0
    value = 2.0 * 2.0 * args.ref_rows * N * K * args.steps / dt / 1e12
    cores = oracle.num_threads()
    sample = (f"each step: {args.ref_rows} of the {M} token rows of the training step (fwd + grad_x through the "
              f"oracle), weights prepared once outside the timing")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "s8",
        "data": "synthetic (seeded splitmix64 + Box-Muller)",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "block": b, "rows_per_step": args.ref_rows},
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["convrot", "reference"], default="convrot")
    ap.add_argument("--cpu-rows", type=int, default=4096, help="token rows in the CPU-oracle sample")
    ap.add_argument("--ref-rows", type=int, default=64, help="token rows per step of --impl reference")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-kernel rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
