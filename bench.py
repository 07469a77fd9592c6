#!/usr/bin/env python3
"""Throughput of the register-tiled product C = A.B on GB300.

One step is one pass of the whole hot path over one batch of synthetic input:
  * gemm_f32      on the fp32 4096 x 4096 x 4096 workload (A, B ~ N(0,1)),
  * gemm_bf16f32  on the bf16 8192 x 8192 x 8192 workload (A, B ~ N(0,1)
                  rounded to bf16), fp32 accumulation and output.
Together they exercise every tiling level of both CUDA paths (global C tiles,
shared-memory K slices, register / tensor-memory accumulator tiles, ragged
edge handling is covered by the tests).

Metric: TFLOP/s = 2*M*N*K summed over the step's products / step time, with
inputs resident in HBM. Each product's own launch duration is timed with CUDA
events on its stream, giving per-kernel TFLOP/s and the roofline fraction
(FP32 SIMT peak for gemm_f32, dense bf16 tensor peak for gemm_bf16f32).
`e2e` repeats the step through the same public calls with host buffers:
pinned host -> device copies of A and B, the product, device -> host copy of C,
every step, pipelined across steps on separate copy streams.

Multi-GPU: the product does not need an exchange, so N GPUs run N independent
replicas (weak scaling); value = all ranks' flops / the slowest rank's time.

--impl reference times the CPU oracle (plain fp64 triple loop) on a bounded
sample of the same workloads, on the host cores.
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
from typing import Dict, List, Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "GEMM TFLOP/s at 1 GB300 and % of FP32-SIMT / bf16-tensor roofline"
UNIT = "TFLOP/s"
STEP = ["f32_4096_normal", "bf16_8192_normal"]
FP32_LANES_PER_SM = 128   # FP32 FMA lanes per Blackwell SM (4 partitions x 32)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# one ncu capture of each kernel, keyed to the kernel source it was taken on;
# reported as null once the source changes.
TRAFFIC = {
    "gemm_f32": {"bytes": 320613632, "source_sha1": "f643ecf29a791456a05c4f2aa30eacb6809e1a1e"},
    "gemm_bf16f32": {"bytes": 1365153024,
                     "source_sha1": "2564a8cd5cb12f0cd75e69661170f865254c938a"},
}
KERNEL_SOURCE = {
    "gemm_f32": "register_tiled_matrix_gb300/csrc/sgemm_tma.cu",  # 4096^3: the TMA-fed tiles
    "gemm_bf16f32": "register_tiled_matrix_gb300/csrc/gemm_tc2.cu",  # M > 128: CTA pairs
}


def source_sha1(kernel: str) -> str:
    with open(os.path.join(ROOT, KERNEL_SOURCE[kernel]), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


def load_peaks() -> Dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


# ------------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def reduce_over_ranks(elapsed_s: float, flops: float, device) -> (float, float):
    """(max elapsed over ranks, sum of flops over ranks); identity at world 1."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return elapsed_s, flops
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    f = torch.tensor([flops], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(f, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(f.item())


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples the SM clock, power and clock-event reasons of one GPU during a
    timed region, read-only: through NVML (libnvidia-ml, every `period_ms`)
    where it loads, else through `nvidia-smi -lms`."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    # NVML clock-event reason bits (nvml.h: nvmlClocksEventReason*)
    NVML_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                 "hw_thermal_slowdown": 0x40}

    def __init__(self, gpu_index: int, period_ms: int = 10, uuid: Optional[str] = None):
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self.uuid = uuid
        self.samples: List[tuple] = []  # (sm_mhz, max_mhz, power_w, reason bits)
        self.lines: List[str] = []
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.source = None

    def _nvml(self):
        import ctypes

        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if nv.nvmlInit_v2() != 0:
            return None
        handle = ctypes.c_void_p()
        ok = False
        if self.uuid:
            for u in (self.uuid, "GPU-" + self.uuid):
                if nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(handle)) == 0:
                    ok = True
                    break
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(self.gpu_index, ctypes.byref(handle)) != 0:
            return None
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or getattr(
            nv, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        return nv, handle, reasons

    def _nvml_loop(self, nv, handle, reasons):
        import ctypes

        sm, mx, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))  # NVML_CLOCK_SM = 1
        try:
            while not self.stop_flag.is_set():
                if nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(sm)) == 0:
                    power = (mw.value / 1e3
                             if nv.nvmlDeviceGetPowerUsage(handle, ctypes.byref(mw)) == 0 else None)
                    bits = (rs.value
                            if reasons is not None and reasons(handle, ctypes.byref(rs)) == 0 else 0)
                    self.samples.append((float(sm.value), float(mx.value), power, bits))
                self.stop_flag.wait(self.period_ms / 1e3)
        finally:
            nv.nvmlShutdown()

    def start(self):
        nvml = None
        try:
            nvml = self._nvml()
        except (OSError, AttributeError):
            nvml = None
        if nvml is not None:
            self.source = f"nvml every {self.period_ms} ms"
            self.thread = threading.Thread(target=self._nvml_loop, args=nvml, daemon=True)
            self.thread.start()
            time.sleep(0.05)
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(max(self.period_ms, 20)), "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.source = f"nvidia-smi every {max(self.period_ms, 20)} ms"
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)  # let the first sample land before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> Dict:
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "neither NVML nor nvidia-smi available"}
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, pw = [], [], []
        active = set()
        for (s_mhz, m_mhz, p_w, bits) in self.samples:
            sm.append(s_mhz)
            mx.append(m_mhz)
            if p_w is not None:
                pw.append(p_w)
            for name, bit in self.NVML_BITS.items():
                if bits & bit:
                    active.add(name)
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower() == "active":
                    active.add(name)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None,
            "sm_mhz_min": min(sm) if sm else None,
            "reasons": sorted(active),
            "samples": len(sm),
            "power_w_median": statistics.median(pw) if pw else None,
            "power_w_max": max(pw) if pw else None,
            "source": self.source,
        }


# ------------------------------------------------------------------ our arm
def make_step_inputs(device, names):
    items = []
    for name in names:
        w = workloads.WORKLOADS[name]
        A, B = workloads.workload_inputs(w)
        items.append({
            "name": name, "w": w,
            "A_host": A.pin_memory(), "B_host": B.pin_memory(),
            "A": A.to(device), "B": B.to(device),
            "C": torch.empty((w.M, w.N), dtype=torch.float32, device=device),
            "C_host": torch.empty((w.M, w.N), dtype=torch.float32).pin_memory(),
        })
    return items


def count_kernel_launches(fn) -> Optional[int]:
    """How many kernels one call of fn launches, counted from the device kernel
    activities (memory copies and sets excluded) the PyTorch profiler records
    for that call. None when the count cannot be taken."""
    try:
        from torch.profiler import ProfilerActivity, profile

        def kernels():
            torch.cuda.synchronize()
            with profile(activities=[ProfilerActivity.CUDA]) as prof:
                fn()
                torch.cuda.synchronize()
            return sum(1 for e in prof.events()
                       if str(getattr(e, "device_type", "")).endswith("CUDA")
                       and not e.name.startswith(("Memcpy", "Memset")))

        kernels()  # the first session may start the tracer after the launches
        n = kernels()
        return n if n > 0 else None
    except Exception:  # a count, not a result: report it as unknown
        return None


def kernel_of(w) -> str:
    return "gemm_f32" if w.dtype == "f32" else "gemm_bf16f32"


def step_names(only: Optional[str]) -> List[str]:
    names = [n for n in STEP if only is None or kernel_of(workloads.WORKLOADS[n]) == only]
    if not names:
        raise SystemExit(f"--only {only}: no such entry point in the step")
    return names


def step_config(names: List[str], world: int) -> Dict:
    parts = []
    for n in names:
        w = workloads.WORKLOADS[n]
        kind = "fp32" if w.dtype == "f32" else "bf16->fp32"
        parts.append(f"{kernel_of(w)} {w.M}x{w.N}x{w.K} {kind}")
    return {
        "workload": "one step = " + " + ".join(parts) + ", row-major, N(0,1) inputs",
        "products": [{"name": n, "M": workloads.WORKLOADS[n].M, "N": workloads.WORKLOADS[n].N,
                      "K": workloads.WORKLOADS[n].K, "entry": kernel_of(workloads.WORKLOADS[n])}
                     for n in names],
        "parallelism": f"replicas x{world} (no exchange)",
        "l2": "no explicit flush: the step's working set of A, B and C exceeds the 129 MB L2 "
              "and each product evicts the other's operands between iterations",
    }


def run_ours(args) -> Optional[Dict]:
    import register_tiled_matrix_gb300 as rtm

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (sm_103a)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    if rank == 0:
        rtm.build()
    barrier()
    rtm.load_library()
    fns = {"gemm_f32": rtm.gemm_f32, "gemm_bf16f32": rtm.gemm_bf16f32}

    names = step_names(args.only)
    items = make_step_inputs(device, names)
    stream = torch.cuda.current_stream(device)
    step_flops = sum(it["w"].flops for it in items)

    def step(record=None):
        for i, it in enumerate(items):
            if record is not None:
                record[i][0].record(stream)
            fns[kernel_of(it["w"])](it["A"], it["B"], out=it["C"])
            if record is not None:
                record[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    if rtm.get_device_error() != 0:
        raise SystemExit("device error during warm-up")

    # ---- timed region: K steps, inputs resident in HBM
    # The FP32 pipes' own throughput on this GPU (the denominator of gemm_f32's
    # roofline), measured before the timed region: independent FMA chains, no
    # memory traffic, scalar and packed forms.
    fp32_measured = None
    if "gemm_f32" in {kernel_of(it["w"]) for it in items} and not args.no_peak:
        fp32_measured = {"scalar": rtm.fp32_pipe_peak(iters=5000, packed=False),
                         "packed": rtm.fp32_pipe_peak(iters=5000, packed=True)}
        torch.cuda.synchronize(device)

    per_kernel = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in items] for _ in range(args.steps)]
    e_all0 = torch.cuda.Event(enable_timing=True)
    e_all1 = torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(device)
    clocks = ClockSampler(torch.cuda.current_device(), uuid=str(getattr(props, "uuid", "") or ""))
    clocks.start()
    barrier()
    torch.cuda.synchronize(device)
    e_all0.record(stream)
    for k in range(args.steps):
        step(per_kernel[k])
    e_all1.record(stream)
    torch.cuda.synchronize(device)
    barrier()
    clock_summary = clocks.stop()
    elapsed_s = e_all0.elapsed_time(e_all1) / 1e3
    dev_err = rtm.get_device_error()
    if dev_err != 0:
        raise SystemExit(f"device error in the timed region: {rtm.status_string(dev_err)}")
    per_call = [count_kernel_launches(
        lambda it=it: fns[kernel_of(it["w"])](it["A"], it["B"], out=it["C"])) for it in items]
    launches = args.steps * sum(n if n is not None else 1 for n in per_call)
    launch_note = {it["name"]: n for it, n in zip(items, per_call)}

    kernel_ms = {}
    for i, it in enumerate(items):
        ts = [per_kernel[k][i][0].elapsed_time(per_kernel[k][i][1]) for k in range(args.steps)]
        kernel_ms[it["name"]] = {"mean": statistics.fmean(ts), "median": statistics.median(ts),
                                 "min": min(ts)}

    # ---- end to end: host buffers, copies inside the timed region
    e2e_steps = 0 if args.no_e2e else args.steps
    h2d = sum(it["A_host"].numel() * it["A_host"].element_size()
              + it["B_host"].numel() * it["B_host"].element_size() for it in items)
    d2h = sum(it["C_host"].numel() * 4 for it in items)

    # Pipelined like a serving loop: the host->device copies of step i+1 and
    # the device->host copy of step i-1 run on their own streams while step i
    # computes; device operands are double-buffered. Every step still moves
    # all of its inputs in and its full C out inside the timed region.
    h2d_stream = torch.cuda.Stream(device)
    d2h_stream = torch.cuda.Stream(device)
    for it in items:
        it["A2"] = [it["A"], torch.empty_like(it["A"])]
        it["B2"] = [it["B"], torch.empty_like(it["B"])]
        it["C2"] = [it["C"], torch.empty_like(it["C"])]
        it["Ch2"] = [it["C_host"], torch.empty_like(it["C_host"]).pin_memory()]
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("h2d", "comp", "d2h")}
    for name in ev:
        for e in ev[name]:
            e.record(stream)

    def step_e2e(i):
        slot = i % 2
        h2d_stream.wait_event(ev["comp"][slot])   # step i-2 no longer reads this slot
        with torch.cuda.stream(h2d_stream):
            for it in items:
                it["A2"][slot].copy_(it["A_host"], non_blocking=True)
                it["B2"][slot].copy_(it["B_host"], non_blocking=True)
        ev["h2d"][slot].record(h2d_stream)
        stream.wait_event(ev["h2d"][slot])
        stream.wait_event(ev["d2h"][slot])        # step i-2's C has left this slot
        for it in items:
            fns[kernel_of(it["w"])](it["A2"][slot], it["B2"][slot], out=it["C2"][slot],
                                    stream=stream)
        ev["comp"][slot].record(stream)
        d2h_stream.wait_event(ev["comp"][slot])
        with torch.cuda.stream(d2h_stream):
            for it in items:
                it["Ch2"][slot].copy_(it["C2"][slot], non_blocking=True)
        ev["d2h"][slot].record(d2h_stream)

    e2e_s = 0.0
    if e2e_steps:
        step_e2e(0)
        step_e2e(1)
        torch.cuda.synchronize(device)
        barrier()
        x0 = torch.cuda.Event(enable_timing=True)
        x1 = torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        h2d_stream.wait_event(x0)
        for i in range(e2e_steps):
            step_e2e(i)
        stream.wait_event(ev["d2h"][(e2e_steps - 1) % 2])  # the last C is on the host
        stream.wait_event(ev["d2h"][e2e_steps % 2])
        x1.record(stream)
        torch.cuda.synchronize(device)
        barrier()
        e2e_s = x0.elapsed_time(x1) / 1e3

    max_elapsed, all_flops = reduce_over_ranks(elapsed_s, step_flops * args.steps, device)
    max_e2e, all_e2e_flops = reduce_over_ranks(e2e_s, step_flops * e2e_steps, device)
    if rank != 0:
        return None

    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    max_mhz = float(peaks.get("sm_max_mhz") or FALLBACK_PEAKS["sm_max_mhz"])
    fp32_derived = sms * FP32_LANES_PER_SM * 2 * max_mhz * 1e6 / 1e12
    # gemm_f32's roofline peak: the faster of the two measured FMA forms (the
    # pipes' own ceiling on this GPU); the derived figure when not measured.
    if fp32_measured is not None:
        fp32_peak = max(fp32_measured["scalar"]["tflops"], fp32_measured["packed"]["tflops"])
        fp32_note = ("measured on this GPU before the timed region: best of scalar and packed "
                     "FP32 FMA chains (gemm_fp32_pipe_peak), "
                     f"{fp32_measured['scalar']['tflops']:.2f} / "
                     f"{fp32_measured['packed']['tflops']:.2f} TFLOP/s at "
                     f"{fp32_measured['scalar']['sm_mhz']:.0f} MHz")
    else:
        fp32_peak = fp32_derived
        fp32_note = (f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x "
                     f"{max_mhz:.0f} MHz")
    # The step alternates an FP32-pipe product with the tensor-core product and
    # does not reach the power cap (the clock record shows it), so the tensor
    # product is compared with the burst bf16 figure; the power-capped
    # sustained figure is reported beside it.
    bf16_peak = float(peaks["bf16_tflops"])
    bf16_sustained = float(peaks.get("bf16_tflops_sustained") or bf16_peak)

    rooflines = {}
    for it in items:
        w = it["w"]
        kern = kernel_of(w)
        ms = kernel_ms[it["name"]]["mean"]
        achieved = w.flops / (ms / 1e3) / 1e12
        if kern == "gemm_f32":
            bound, peak, peak_note = "alu", fp32_peak, fp32_note
        else:
            bound, peak, peak_note = "tensor", bf16_peak, (
                f"{peaks['source']} dense bf16 burst (cuBLAS 8192^3); clocks stay at max in "
                f"this step")
        traffic = TRAFFIC[kern]
        tb = traffic["bytes"] if traffic["source_sha1"] == source_sha1(kern) else None
        rooflines[kern] = {
            "bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 2),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": tb,
            "peak_source": peak_note, "workload": it["name"],
            "ms_mean": round(ms, 4), "ms_median": round(kernel_ms[it["name"]]["median"], 4),
            "algorithmic_flops": w.flops,
            "algorithmic_bytes": w.in_bytes + w.out_bytes,
        }
        if kern == "gemm_bf16f32":
            rooflines[kern]["frac_of_sustained"] = round(achieved / bf16_sustained, 4)
        else:
            rooflines[kern]["frac_of_derived"] = round(achieved / fp32_derived, 4)
            if fp32_measured is not None:
                rooflines[kern]["frac_of_scalar_ffma"] = round(
                    achieved / fp32_measured["scalar"]["tflops"], 4)
    dominant = max(items, key=lambda it: kernel_ms[it["name"]]["mean"])
    out = {
        "metric": METRIC,
        "value": round(all_flops / max_elapsed / 1e12, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_elapsed * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 (gemm_f32) + bf16 in / f32 accumulate (gemm_bf16f32)",
        "data": "synthetic (seeded N(0,1); bf16 inputs rounded to nearest even)",
        "config": step_config(names, world),
        "roofline": rooflines[kernel_of(dominant["w"])],
        "rooflines": rooflines,
        "kernel_ms": {k: {kk: round(vv, 4) for kk, vv in v.items()} for k, v in kernel_ms.items()},
        "e2e": ({"value": round(all_e2e_flops / max_e2e / 1e12, 3), "unit": UNIT,
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}
                if e2e_steps else None),
        "gpu_launches": launches,
        "gpu_launches_per_call": launch_note,
        "clocks": clock_summary,
        "peaks": {"source": peaks["source"], "fp32_simt_tflops": round(fp32_peak, 2),
                  "fp32_simt_tflops_measured": (round(fp32_peak, 2) if fp32_measured else None),
                  "fp32_scalar_ffma_tflops_measured": (
                      round(fp32_measured["scalar"]["tflops"], 2) if fp32_measured else None),
                  "fp32_packed_ffma_tflops_measured": (
                      round(fp32_measured["packed"]["tflops"], 2) if fp32_measured else None),
                  "fp32_peak_sm_mhz": (round(fp32_measured["scalar"]["sm_mhz"], 1)
                                       if fp32_measured else None),
                  "fp32_simt_tflops_derived": round(fp32_derived, 2),
                  "bf16_tflops_burst": bf16_peak, "bf16_tflops_sustained": bf16_sustained},
    }
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(names, items, budget_s=args.cpu_budget)
    return out


# ------------------------------------------------------------------ oracle timing
def _oracle_inputs(names, items=None):
    import numpy as np

    res = []
    for name in names:
        w = workloads.WORKLOADS[name]
        if items is not None:
            it = next(x for x in items if x["name"] == name)
            A, B = it["A_host"], it["B_host"]
        else:
            A, B = workloads.workload_inputs(w)
        res.append((w, np.ascontiguousarray(A.float().numpy()),
                    np.ascontiguousarray(B.float().numpy())))
    return res


def _oracle_sample(oracle, w, A, B, count, seed):
    rows, cols = workloads.sample_indices(w.M, w.N, count=count, seed=seed, edge_count=0)
    rows, cols = rows[:count], cols[:count]
    t0 = time.perf_counter()
    oracle.gemm_sampled(A, B, rows, cols)
    return time.perf_counter() - t0, 2.0 * w.K * len(rows)


def _calibrate(oracle, inputs, probe=256):
    """Seconds per sampled entry of each product (entries split over all threads)."""
    rates = []
    for (w, A, B) in inputs:
        dt, _ = _oracle_sample(oracle, w, A, B, probe, seed=w.seed)
        rates.append(dt / probe)
    return rates


def cpu_baseline(names, items=None, budget_s: float = 15.0) -> Dict:
    """Time the oracle as it stands on a bounded sample of the step's products."""
    import oracle

    oracle.build()
    inputs = _oracle_inputs(names, items)
    per_entry = _calibrate(oracle, inputs)
    share = budget_s / len(inputs)
    total_t, total_f, desc = 0.0, 0.0, []
    for (w, A, B), pe in zip(inputs, per_entry):
        count = max(oracle.max_threads(), int(share / max(pe, 1e-9)))
        dt, fl = _oracle_sample(oracle, w, A, B, count, seed=w.seed + 7)
        total_t += dt
        total_f += fl
        desc.append(f"{count} seeded entries of C for {w.name}")
    return {"value": total_f / total_t / 1e12, "unit": UNIT, "cores": oracle.max_threads(),
            "cpu_model": cpu_model(), "kind": "oracle",
            "sample": "; ".join(desc) + f" (fp64 dot products of length K, {total_t:.1f} s)"}


def run_reference(args) -> Optional[Dict]:
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle

    oracle.build()
    names = step_names(args.only)
    inputs = _oracle_inputs(names)
    per_entry = _calibrate(oracle, inputs)
    steps_total = args.steps + args.warmup
    per_step_budget = args.reference_budget / max(steps_total, 1)
    counts = [max(1, int(per_step_budget / len(inputs) / max(pe, 1e-9))) for pe in per_entry]
    for i in range(args.warmup):
        for (w, A, B), c in zip(inputs, counts):
            _oracle_sample(oracle, w, A, B, c, seed=w.seed + 100 + i)
    total_t, total_f = 0.0, 0.0
    for k in range(args.steps):
        for (w, A, B), c in zip(inputs, counts):
            dt, fl = _oracle_sample(oracle, w, A, B, c, seed=w.seed + 1000 + k)
            total_t += dt
            total_f += fl
    value = total_f / total_t / 1e12
    sample = "per step: " + "; ".join(
        f"{c} seeded entries of C for {w.name}" for (w, _, _), c in zip(inputs, counts))
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_t * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle accumulation)",
        "data": "synthetic (seeded N(0,1); bf16 inputs rounded to nearest even)",
        "config": step_config(names, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "cpu_model": cpu_model(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ladder(args) -> Optional[Dict]:
    """Time the page's ablation ladder (gemm_f32_ladder rungs 0-6) on one square size."""
    import register_tiled_matrix_gb300 as rtm
    from oracle import tiling_model

    if not torch.cuda.is_available():
        raise SystemExit("bench.py --ladder needs a CUDA GPU (sm_103a)")
    rtm.build()
    n = args.ladder_size
    A, B = workloads.make_inputs(n, n, n, "normal", "f32", seed=workloads.SEED_BASE + 99)
    A, B = A.cuda(), B.cuda()
    C = torch.empty(n, n, device="cuda")
    flops = 2.0 * n ** 3
    # Model of shared reads per output per k for each rung (counting model of
    # the page's loops): naive 0, shared-tiled 2, T x T register tile 2/T.
    reads = tiling_model.predicted_shared_reads_per_output_per_k
    model = {0: 0.0, 1: 2.0, 2: reads(4, 4), 3: reads(8, 8), 4: reads(1, 1), 5: reads(2, 2),
             6: reads(8, 8)}
    rungs = []
    for rung in range(7):
        for _ in range(args.warmup):
            rtm.gemm_f32_ladder(rung, A, B, out=C)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            rtm.gemm_f32_ladder(rung, A, B, out=C)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        rungs.append({"rung": rung, "kernel": rtm.LADDER[rung], "ms": round(ms, 4),
                      "tflops": round(flops / ms / 1e9, 2),
                      "model_shared_reads_per_output_per_k": model[rung]})
    if rtm.get_device_error() != 0:
        raise SystemExit("device error in the ladder")
    return {"metric": "ablation ladder: GEMM TFLOP/s per tiling level", "unit": UNIT,
            "config": {"workload": f"gemm_f32_ladder {n}x{n}x{n} fp32, N(0,1) inputs"},
            "steps": args.steps, "warmup": args.warmup, "rungs": rungs}


def run_configs(args) -> Optional[Dict]:
    """Time every configuration's product (report only; the headline is the step)."""
    import register_tiled_matrix_gb300 as rtm

    if not torch.cuda.is_available():
        raise SystemExit("bench.py --configs needs a CUDA GPU (sm_103a)")
    rtm.build()
    peaks = load_peaks()
    props = torch.cuda.get_device_properties(0)
    sms = props.multi_processor_count
    fp32_derived = sms * FP32_LANES_PER_SM * 2 * float(peaks.get("sm_max_mhz") or 2070.0) * 1e6 / 1e12
    fp32_measured = {"scalar": rtm.fp32_pipe_peak(iters=5000, packed=False),
                     "packed": rtm.fp32_pipe_peak(iters=5000, packed=True)}
    fp32_peak = max(fp32_measured["scalar"]["tflops"], fp32_measured["packed"]["tflops"])
    hbm = float(peaks.get("hbm_gbs") or 6800.0)
    rows = []
    oracle_rows = []
    # L2-cold timing: before each timed call, write a buffer twice the L2's size
    # (outside the timed interval), so the call finds none of its operands in L2.
    l2_bytes = int(getattr(props, "L2_cache_size", 0) or (129 << 20))
    flush = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device="cuda")

    def timed_cold(fn, reps=None):
        reps = reps or max(3, min(args.steps, 20))
        for _ in range(2):
            fn()
        ts = []
        for _ in range(reps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    def timed_graph(fn):
        """Per-call time with the calls replayed from a CUDA graph: the device
        time without the binding's host cost per call, which bounds small
        products called back to back from Python. None if capture fails."""
        calls = max(1, min(args.steps, 20))
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                fn()  # per-device caches filled outside the capture
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(calls):
                    fn()
            graph.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            reps = 3
            e0.record()
            for _ in range(reps):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / (reps * calls)
        except RuntimeError:
            torch.cuda.synchronize()
            return None

    if args.shapes:
        todo = []
        for i, spec in enumerate(args.shapes.split(",")):
            dims, _, dt = spec.partition(":")
            M, N, K = (int(x) for x in dims.split("x"))
            dt = dt or "f32"
            todo.append(workloads.Workload(f"{dt}_{M}x{N}x{K}", M, N, K, dt, "normal",
                                           workloads.SEED_BASE + 1000 + i, False))
    else:
        names = args.config_names.split(",") if args.config_names else list(workloads.WORKLOADS)
        todo = [workloads.WORKLOADS[name] for name in names]
    for w in todo:
        name = w.name
        A, B = workloads.workload_inputs(w)
        A, B = A.cuda(), B.cuda()
        C = torch.empty(w.M, w.N, device="cuda")
        entries = []
        if w.dtype == "f32":
            kind, splits = rtm.gemm_f32_schedule(w.M, w.N, w.K)
            label = "gemm_f32" if kind == "tiles" else f"gemm_f32 ({kind} x{splits})"
            entries.append((label, lambda: rtm.gemm_f32(A, B, out=C), fp32_peak))
            need = rtm.gemm_f32_workspace_bytes(w.M, w.N, w.K)
            if need > 0:
                ws = torch.empty(need // 4, device="cuda")
                wkind, wsplits = rtm.gemm_f32_schedule(w.M, w.N, w.K, workspace=True)
                entries.append((f"gemm_f32_ws ({wkind} x{wsplits})",
                                lambda: rtm.gemm_f32_ws(A, B, out=C, workspace=ws), fp32_peak))
        else:
            entries.append(("gemm_bf16f32", lambda: rtm.gemm_bf16f32(A, B, out=C),
                            float(peaks["bf16_tflops"])))
            # Rows off 16-byte boundaries: with M > 128 the workspace entry
            # re-pitches them for the TMA-fed CTA pairs; with M <= 128, and for
            # tall, narrow products with long K (N <= 128, at least 32 64-deep
            # K-blocks, the 128-row tiles fitting on the SMs), it runs the same
            # kernel as gemm_bf16f32 and is not timed again.
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            cols = 64 if w.N <= 64 else 128
            tall_narrow = (w.N <= 128 and (w.K + 63) // 64 >= 32 and
                           (w.M + 127) // 128 * ((w.N + cols - 1) // cols) <= sms)
            if (w.K % 8 or w.N % 8) and w.M > 128 and not tall_narrow:
                wsb = torch.empty(rtm.gemm_bf16f32_workspace_bytes(w.M, w.N, w.K),
                                  dtype=torch.uint8, device="cuda")
                entries.append(("gemm_bf16f32_ws (rows re-pitched, CTA pairs)",
                                lambda: rtm.gemm_bf16f32_ws(A, B, out=C, workspace=wsb),
                                float(peaks["bf16_tflops"])))
        for entry, fn, peak in entries:
            ms = timed(fn)
            ms_cold = timed_cold(fn)
            ms_graph = timed_graph(fn)
            tf = w.flops / ms / 1e9
            # Binding roofline of this product: the larger of its compute time
            # at the peak and its algorithmic bytes at the measured copy bandwidth.
            alg_bytes = w.in_bytes + w.out_bytes
            t_compute = w.flops / (peak * 1e12) * 1e3
            t_memory = alg_bytes / (hbm * 1e9) * 1e3
            roof_ms = max(t_compute, t_memory)
            rows.append({"config": name, "M": w.M, "N": w.N, "K": w.K, "entry": entry,
                         "ms": round(ms, 4), "tflops": round(tf, 2),
                         "frac_of_peak": round(tf / peak, 4),
                         "l2_cold_ms": round(ms_cold, 4),
                         "l2_cold_tflops": round(w.flops / ms_cold / 1e9, 2),
                         "bound": "compute" if t_compute >= t_memory else "hbm",
                         "roof_ms": round(roof_ms, 4), "frac_of_roofline": round(roof_ms / ms, 4),
                         "ms_graph": None if ms_graph is None else round(ms_graph, 4),
                         "frac_of_roofline_graph": (None if ms_graph is None
                                                    else round(roof_ms / ms_graph, 4))})
        if not args.no_oracle and not args.shapes:
            oracle_rows.append(oracle_timing(w))
        del A, B, C
        torch.cuda.empty_cache()
    if rtm.get_device_error() != 0:
        raise SystemExit("device error in the configs run")
    out = {"metric": "GEMM TFLOP/s per configuration (report only)", "unit": UNIT,
           "steps": args.steps, "warmup": args.warmup,
           "peaks": {"fp32_simt_tflops": round(fp32_peak, 2),
                     "fp32_simt_tflops_source": "measured (gemm_fp32_pipe_peak, best of scalar "
                                                "and packed FMA chains)",
                     "fp32_scalar_ffma_tflops_measured": round(fp32_measured["scalar"]["tflops"], 2),
                     "fp32_packed_ffma_tflops_measured": round(fp32_measured["packed"]["tflops"], 2),
                     "fp32_simt_tflops_derived": round(fp32_derived, 2),
                     "bf16_tflops_burst": float(peaks["bf16_tflops"]), "hbm_gbs": hbm},
           "l2": ("ms: back-to-back launches (L2-warm for the smaller configs); l2_cold_ms: "
                  f"median of single launches, each after writing {2 * l2_bytes >> 20} MiB "
                  "(twice the L2) outside the timed interval"),
           "configs": rows}
    if oracle_rows:
        out["oracle"] = {"cpu_model": cpu_model(), "cores": _oracle_cores(), "rows": oracle_rows}
    return out


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def _oracle_cores() -> int:
    import oracle

    oracle.build()
    return oracle.max_threads()


# Products the oracle multiplies in full when timed (M*N*K <= 2^31); larger
# ones are timed on sampled entries and extrapolated to the full product by
# their rate per multiply-add.
ORACLE_FULL_MACS = 1 << 31


def oracle_timing(w, sample_count: int = 4096) -> Dict:
    """The oracle, as it stands, on one configuration: one thread and all host
    cores; the whole product where M*N*K <= 2^31, else sampled entries of C
    with the full-product time extrapolated from their rate."""
    import oracle

    oracle.build()
    A, B = workloads.workload_inputs(w)
    macs = w.M * w.N * w.K
    row = {"config": w.name, "M": w.M, "N": w.N, "K": w.K, "cores": oracle.max_threads()}
    if macs <= ORACLE_FULL_MACS:
        for label, threads in (("one_thread_s", 1), ("all_cores_s", 0)):
            t0 = time.perf_counter()
            oracle.gemm(A, B, threads=threads)
            row[label] = round(time.perf_counter() - t0, 4)
        row["kind"] = "full product"
    else:
        rows_i, cols_i = workloads.sample_indices(w.M, w.N, count=sample_count, seed=w.seed + 5,
                                                  edge_count=0)
        rows_i, cols_i = rows_i[:sample_count], cols_i[:sample_count]
        sampled_macs = len(rows_i) * w.K
        for label, threads in (("one_thread_s", 1), ("all_cores_s", 0)):
            t0 = time.perf_counter()
            oracle.gemm_sampled(A, B, rows_i, cols_i, threads=threads)
            dt = time.perf_counter() - t0
            row[label + "_sampled"] = round(dt, 4)
            row[label] = round(dt * macs / sampled_macs, 2)
        row["kind"] = (f"extrapolated from {len(rows_i)} sampled entries of C "
                       "(time per multiply-add x M*N*K)")
    return row


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    p.add_argument("--no-peak", action="store_true",
                   help="skip the FP32 pipe measurement (gemm_f32's roofline then uses the "
                        "derived peak)")
    p.add_argument("--only", choices=["gemm_f32", "gemm_bf16f32"], default=None,
                   help="time one entry point's product instead of the whole step")
    p.add_argument("--cpu-budget", type=float, default=15.0,
                   help="seconds of oracle work for the cpu_baseline sample")
    p.add_argument("--reference-budget", type=float, default=120.0,
                   help="seconds of oracle work for the whole --impl reference run")
    p.add_argument("--ladder", action="store_true",
                   help="time the ablation ladder (gemm_f32_ladder rungs 0-3) instead of the step")
    p.add_argument("--ladder-size", type=int, default=4096)
    p.add_argument("--configs", action="store_true",
                   help="time every configuration's product (report only)")
    p.add_argument("--config-names", default=None,
                   help="comma-separated workload names for --configs (default: all)")
    p.add_argument("--no-oracle", action="store_true",
                   help="--configs without the oracle's CPU timings")
    p.add_argument("--shapes", default=None,
                   help="--configs on these products instead, e.g. 16x8192x8192:bf16,4096x4096x4096:f32")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    world, rank, _ = dist_env()
    if args.gpus != world and not (world == 1 and args.gpus == 1):
        if world == 1:
            p.error(f"--gpus {args.gpus} needs torchrun with --nproc-per-node {args.gpus}")
    if args.ladder:
        out = run_ladder(args)
    elif args.configs:
        out = run_configs(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
