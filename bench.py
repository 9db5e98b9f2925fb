#!/usr/bin/env python3
"""Benchmark of the fine-grained FP8 GEMM path on B300.

One step = one FP8 forward of a linear layer at M=4096, N=4096, K=7168 from
bf16 inputs already resident in HBM: activation quantization (1x128 tiles)
and weight quantization (128x128 blocks) in one launch, then the block-scaled
GEMM with bf16 output. The headline value is GEMM FLOPs over the whole step's time
(TFLOP/s). The same run also measures, as extra keys:

* the small reference case (M=128, N=256, K=512) in microseconds,
* the activation quantizer alone on [16384, 7168] with 0.5% outlier channels
  (GB/s against the HBM roofline),
* RMSNorm (and LayerNorm with beta) fused with the 1x128 cast on the same
  [16384, 7168] shape,
* the headline step with the activation quantization inside the GEMM kernel,
* the GEMM M=4096, N=7168, K=2048 with 0.5% outlier channels x50, alone and
  after the quantization of its operands,
* the MoE grouped GEMM (32 experts, N=4096, K=7168, seeded top-8 routing),
* the end-to-end step from pinned host buffers (`e2e`),
* the CPU oracle on a bounded sample (`cpu_baseline`).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--part all|step|small|act_quant|norm_quant|fused|gemm2|moe] [--skip-cpu]

With --gpus N > 1 (launched by torchrun) every rank runs the same step on its
own GPU with no collective on the data path (independent replicas, weak
scaling); the value is the sum of all ranks' work over the slowest rank's time.
`--impl reference` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_fine_grained_17_b300 import workloads as wl  # noqa: E402

L2_BYTES = 126 * 2 ** 20
METRIC = "FP8 block-scaled GEMM TFLOP/s (% of dense FP8 peak); act-quant HBM GB/s"
UNIT = "TFLOP/s"
WORKLOAD = ("GEMM M=4096,N=4096,K=7168: A bf16 ~N(0,1), W bf16 ~N(0,0.02), "
            "block-quantized to E4M3, bf16 out")
M3, N3, K3 = 4096, 4096, 7168
EVENT_EVERY = 8   # timed steps per step with per-kernel events (headline step)
CSRC = os.path.join(ROOT, "fp8_fine_grained_17_b300", "csrc")

# DRAM bytes (read + write) per launch from one ncu capture of each kernel,
# keyed by the SHA-256 prefix of the kernel's source file at capture time. A
# kernel whose source has changed since reports traffic = null.
NCU_TRAFFIC = {
    # kernel: (source file, sha256 prefix, workload, bytes per launch)
    "fp8_gemm_kernel": ("fp8bs_gemm.cu", "308faa69d74c6898", "gemm 4096x4096x7168",
                        60.821760e6 + 16.235776e6),
    "quantize_ring_kernel": ("fp8bs_quant.cu", "d89de783f9cb05b6", "act-quant 16384x7168",
                             234.969088e6 + 78.782208e6),
    "norm_quant_kernel": ("fp8bs_norm.cu", "e5d0f7cd94013121", "norm-quant 16384x7168",
                          237.028608e6 + 66.420224e6),
}


def _src_hash(fname: str) -> str:
    with open(os.path.join(CSRC, fname), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _traffic(kernel: str, workload: str):
    ent = NCU_TRAFFIC.get(kernel)
    if ent is None or ent[2] != workload or _src_hash(ent[0]) != ent[1]:
        return None
    return ent[3]


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def _fp8_peak(peaks):
    """Dense FP8 peak: measured bf16 cuBLAS burst x the nominal FP8/BF16 ratio
    (4.5 / 2.25 PFLOP/s)."""
    return peaks["bf16_tflops"] * 2.0


class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi while it
    is open (one line every 50 ms). Entering waits (up to 10 s) for the first
    sample, so a short timed region is never missed while nvidia-smi starts;
    callers keep the GPU busy with the same work for at least MIN_WINDOW_S
    after the timed region so that the record holds samples under load."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    NAMED = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    MIN_WINDOW_S = 1.0

    def __init__(self, device: torch.device, period_ms: int = 50):
        self.cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", f"-lms={period_ms}"]
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.cmd.append("--id=" + (uuid if uuid.startswith("GPU-") else "GPU-" + uuid))
        except Exception:
            pass
        self.proc = None
        self.lines = []
        self._thread = None
        self._first = None
        self.t_start = time.monotonic()

    def _read(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.lines.append(ln.strip())
                self._first.set()

    def __enter__(self):
        import threading
        self._first = threading.Event()
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            self._thread = threading.Thread(target=self._read, daemon=True)
            self._thread.start()
            self._first.wait(timeout=10.0)
        self.t_start = time.monotonic()
        return self

    def elapsed(self) -> float:
        return time.monotonic() - self.t_start

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            if self._thread is not None:
                self._thread.join(timeout=10)

    def summary(self):
        mhz, max_mhz, watts, reasons = [], None, [], set()
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) != len(self.FIELDS):
                continue
            try:
                cur, mx, w = float(f[0]), float(f[1]), float(f[2])
            except ValueError:
                continue
            mhz.append(cur)
            max_mhz = mx
            watts.append(w)
            for name, val in zip(self.NAMED, f[4:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max_mhz,
                "sm_mhz_min": min(mhz) if mhz else None,
                "power_w_max": max(watts) if watts else None,
                "reasons": sorted(reasons), "samples": len(mhz),
                "source": f"nvidia-smi -lms 50 over warm-up, the timed region and at least "
                          f"{self.MIN_WINDOW_S:g} s of the same step after it"}


def keep_busy(clk: "ClockSampler", stream, step, start: int):
    """Runs untimed copies of `step` until the sampler has been open for
    MIN_WINDOW_S, so that its record holds samples under the timed load."""
    i = start
    while clk.elapsed() < clk.MIN_WINDOW_S:
        with torch.cuda.stream(stream):
            for _ in range(16):
                step(i)
                i += 1
        stream.synchronize()


def line_config(world: int) -> dict:
    """The workload both arms' lines name (identical keys and values)."""
    return {"workload": WORKLOAD, "M": M3, "N": N3, "K": K3, "out": "bf16",
            "step": "quantize A 1x128 + quantize W 128x128 + block-scaled GEMM",
            "l2": "inputs larger than L2 (seeded sets rotated, > 126 MB), no flush",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def max_over_ranks(elapsed_ms: float, world: int, device) -> float:
    """The slowest rank's time (every rank gets it), then a barrier; the
    value itself with one rank. Replicas share no data, so this max and the
    timing barriers are the only collectives."""
    if world <= 1:
        return elapsed_ms
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, elapsed_ms: float) -> float:
    """All ranks' work over the slowest rank's time (weak scaling: each rank
    runs the same step on its own GPU)."""
    return world * flops_per_step * steps / (elapsed_ms * 1e-3) / 1e12


def _events(n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def _median_ms(evs):
    return float(np.median([a.elapsed_time(b) for a, b in evs]))


# --------------------------------------------------------------------- our arm

def _dense_inputs(n_sets: int, dev, cfg):
    """n_sets independent seeded (A, W) bf16 pairs on the device."""
    sets = []
    for i in range(n_sets):
        d = cfg(seed=i)
        sets.append((wl.bits_to_torch(d.a_bits).to(dev), wl.bits_to_torch(d.w_bits).to(dev)))
    return sets


def bench_step(fp8bs, dev, stream, peaks, args, world):
    """The headline: quantize A + quantize W + GEMM at 4096 x 4096 x 7168."""
    step_in_bytes = 2 * (M3 * K3 + N3 * K3)
    n_sets = max(2, -(-3 * L2_BYTES // step_in_bytes))
    sets = _dense_inputs(n_sets, dev, wl.cfg3)
    qa = torch.empty((M3, K3), dtype=torch.uint8, device=dev)
    sa = torch.empty((M3, K3 // 128), dtype=torch.float32, device=dev)
    qw = torch.empty((N3, K3), dtype=torch.uint8, device=dev)
    sw = torch.empty((N3 // 128, K3 // 128), dtype=torch.float32, device=dev)
    c = torch.empty((M3, N3), dtype=torch.bfloat16, device=dev)
    ws = fp8bs.workspace(M3, N3, K3, device=dev)   # the GEMM splits its last wave of tiles

    # The two quantizations are independent and run as one launch
    # (fp8bs_quantize_act_and_weight); the GEMM follows on the same stream.
    def step(i, ev=None):
        a, w = sets[i % n_sets]
        if ev is not None:
            ev[0].record(stream)
        fp8bs.fp8bs_quantize_act_and_weight(a, qa, sa, w, qw, sw, stream)
        if ev is not None:
            ev[1].record(stream)
        fp8bs.fp8bs_gemm_ws(qa, sa, qw, sw, c, ws, stream)
        if ev is not None:
            ev[2].record(stream)

    # Per-kernel durations come from events around the two launches of every
    # EVENT_EVERY-th timed step. An event between two kernels makes the second
    # wait for the first to drain before it launches, so recording them on
    # every step would add that gap to every step of the headline.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] if i % EVENT_EVERY == 0 else None
           for i in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        with torch.cuda.stream(stream):
            for i in range(args.warmup):
                step(i)
        stream.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(args.steps):
                step(i, evs[i])
            t1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        keep_busy(clk, stream, step, args.steps)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    assert fp8bs.fp8bs_last_device_error(stream) == fp8bs.OK

    per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])] for e in evs if e is not None])
    t_quant, t_gemm = per.mean(axis=0)
    flops = 2.0 * M3 * N3 * K3
    fp8_peak = _fp8_peak(peaks)
    gemm_tflops = flops / (t_gemm * 1e-3) / 1e12
    qa_bytes = M3 * K3 * 2 + M3 * K3 + M3 * (K3 // 128) * 4
    qw_bytes = N3 * K3 * 2 + N3 * K3 + (N3 // 128) * (K3 // 128) * 4
    del sets
    return {
        "elapsed_ms": elapsed_ms,
        "value": whole_job_tflops(flops, args.steps, world, elapsed_ms),
        "n_sets": n_sets, "set_bytes": n_sets * step_in_bytes,
        "roofline": {"bound": "tensor", "kernel": "fp8_gemm_kernel<2,256> (CTA pair, 256x256 tiles, last wave split)",
                     "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                     "traffic": _traffic("fp8_gemm_kernel", "gemm 4096x4096x7168"),
                     "algorithmic": f"2*M*N*K = {flops:.4g} flop per launch / mean launch time "
                                    f"{t_gemm * 1e3:.2f} us (CUDA events around {len(per)} of the "
                                    f"{args.steps} timed launches, every {EVENT_EVERY}th step)",
                     "peak_note": f"of {peaks['source']}: bf16 cuBLAS burst "
                                  f"{peaks['bf16_tflops']} x 2 (nominal fp8/bf16)",
                     "frac_of_nominal_4500": round(gemm_tflops / 4500.0, 4)},
        "kernels": {
            "quantize_act_and_weight": {
                "us": round(t_quant * 1e3, 2),
                "GB/s": round((qa_bytes + qw_bytes) / (t_quant * 1e-3) / 1e9, 1),
                "frac_hbm": round((qa_bytes + qw_bytes) / (t_quant * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "algorithmic": "A and W: 2 B read + 1 B code per element, 4 B per scale"},
            "gemm": {"us": round(t_gemm * 1e3, 2), "TFLOP/s": round(gemm_tflops, 1)},
        },
        "clocks": clk.summary(),
    }


def bench_fused(fp8bs, dev, stream, peaks, args):
    """The headline workload with the activation quantization inside the GEMM
    kernel: quantize W + fused GEMM(bf16 A) per step, on the same rotated
    input sets; beside it the unfused pair (quantize A, GEMM) on the same
    inputs, timed the same way."""
    step_in_bytes = 2 * (M3 * K3 + N3 * K3)
    n_sets = max(2, -(-3 * L2_BYTES // step_in_bytes))
    sets = _dense_inputs(n_sets, dev, wl.cfg3)
    qa = torch.empty((M3, K3), dtype=torch.uint8, device=dev)
    sa = torch.empty((M3, K3 // 128), dtype=torch.float32, device=dev)
    qw = torch.empty((N3, K3), dtype=torch.uint8, device=dev)
    sw = torch.empty((N3 // 128, K3 // 128), dtype=torch.float32, device=dev)
    c = torch.empty((M3, N3), dtype=torch.bfloat16, device=dev)
    ws = fp8bs.workspace(M3, N3, K3, device=dev)
    n = max(20, min(args.steps, 400))

    def run(fused):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup) + n):
                a, w = sets[i % n_sets]
                ev = evs[i - max(3, args.warmup)] if i >= max(3, args.warmup) else None
                if ev is not None:
                    ev[0].record(stream)
                fp8bs.fp8bs_quantize_weight_128x128(w, qw, sw, stream)
                if ev is not None:
                    ev[1].record(stream)
                if fused:
                    fp8bs.fp8bs_gemm_bf16_act(a, qw, sw, c, stream)
                else:
                    fp8bs.fp8bs_quantize_act_1x128(a, qa, sa, stream)
                    fp8bs.fp8bs_gemm_ws(qa, sa, qw, sw, c, ws, stream)
                if ev is not None:
                    ev[2].record(stream)
        stream.synchronize()
        per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])] for e in evs if e is not None])
        return per.mean(axis=0)

    flops = 2.0 * M3 * N3 * K3
    res = {}
    for rnd in range(2):   # interleaved, two rounds each
        for fused in (True, False):
            res.setdefault(fused, []).append(run(fused))
    assert fp8bs.fp8bs_last_device_error(stream) == fp8bs.OK
    f_qw, f_g = np.mean(res[True], axis=0)
    u_qw, u_g = np.mean(res[False], axis=0)
    del sets
    return {"workload": "GEMM M=4096,N=4096,K=7168 bf16 A, activation 1x128 quantization "
                        "inside the GEMM kernel; step = quantize W + fused GEMM",
            "step_TFLOP/s": round(flops / ((f_qw + f_g) * 1e-3) / 1e12, 1),
            "fused_gemm_us": round(f_g * 1e3, 2),
            "fused_gemm_TFLOP/s": round(flops / (f_g * 1e-3) / 1e12, 1),
            "unfused_step_TFLOP/s": round(flops / ((u_qw + u_g) * 1e-3) / 1e12, 1),
            "unfused_quantA_plus_gemm_us": round(u_g * 1e3, 2),
            "timing": f"mean of {n} steps x 2 interleaved rounds per variant, "
                      f"inputs rotated over {n_sets} sets"}


def bench_act_quant(fp8bs, dev, stream, peaks, args):
    """Activation quantizer alone on [16384, 7168] with 0.5% outlier channels
    x100, alternating between two seeded inputs (470 MB > L2)."""
    xs = [wl.bits_to_torch(wl.cfg1(s).a_bits).to(dev) for s in (0, 1)]
    M, K = xs[0].shape
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            fp8bs.fp8bs_quantize_act_1x128(xs[i % 2], q, s, stream)
    n = max(20, min(args.steps, 200))
    evs = _events(n)
    with torch.cuda.stream(stream):
        for i, (e0, e1) in enumerate(evs):
            e0.record(stream)
            fp8bs.fp8bs_quantize_act_1x128(xs[i % 2], q, s, stream)
            e1.record(stream)
    stream.synchronize()
    ms = _median_ms(evs)
    groups = M * (K // 128)
    nbytes = groups * (256 + 128 + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "act-quant [16384,7168] bf16, 36 outlier channels x100",
            "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "bytes": nbytes,
            "roofline": {"bound": "hbm", "kernel": "quantize_ring_kernel",
                         "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": _traffic("quantize_ring_kernel", "act-quant 16384x7168"),
                         "algorithmic": f"{groups} groups x 388 B (256 B read, 128 B codes, "
                                        f"4 B scale)",
                         "peak_note": f"of {peaks['source']} copy bandwidth",
                         "frac_of_8000": round(gbs / 8000.0, 4)},
            "l2": "two 235 MB inputs alternated (> 126 MB L2)",
            "timing": f"median of {n} launches"}


def bench_norm_quant(fp8bs, dev, stream, peaks, args):
    """RMSNorm fused with the 1x128 cast on [16384, 7168] (0.5% outlier
    channels x100), alternating between two seeded inputs (470 MB > L2).
    LayerNorm with beta on the same inputs is timed beside it (it also writes
    the row means and reads beta)."""
    ns = [wl.norm(16384, 7168, seed=s, with_beta=True) for s in (0, 1)]
    xs = [wl.bits_to_torch(n.x_bits).to(dev) for n in ns]
    g = wl.bits_to_torch(ns[0].gamma_bits).to(dev)
    b = wl.bits_to_torch(ns[0].beta_bits).to(dev)
    M, K = xs[0].shape
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    mean = torch.empty(M, dtype=torch.float32, device=dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    n = max(20, min(args.steps, 200))

    def time_kind(kind, beta, mean_out):
        def call(i):
            fp8bs.fp8bs_norm_quantize_act_1x128(xs[i % 2], g, beta, kind, 1e-6, q, s,
                                                mean_out, rstd, stream)
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup)):
                call(i)
        evs = _events(n)
        with torch.cuda.stream(stream):
            for i, (e0, e1) in enumerate(evs):
                e0.record(stream)
                call(i)
                e1.record(stream)
        stream.synchronize()
        return _median_ms(evs)
    ms = time_kind(fp8bs.NORM_RMS, None, None)
    ms_ln = time_kind(fp8bs.NORM_LAYER, b, mean)
    groups = M * (K // 128)
    nbytes = groups * (256 + 128 + 4) + M * 4 + K * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    nbytes_ln = nbytes + M * 4 + K * 2
    return {"workload": "RMSNorm + act-quant [16384,7168] bf16, 36 outlier channels x100",
            "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "bytes": nbytes,
            "roofline": {"bound": "hbm", "kernel": "norm_quant_kernel",
                         "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "traffic": _traffic("norm_quant_kernel", "norm-quant 16384x7168"),
                         "algorithmic": f"{groups} groups x 388 B (256 B read, 128 B codes, "
                                        f"4 B scale) + 4 B rstd per row + gamma",
                         "peak_note": f"of {peaks['source']} copy bandwidth"},
            "layer_norm_beta": {"us": round(ms_ln * 1e3, 2),
                                "GB/s": round(nbytes_ln / (ms_ln * 1e-3) / 1e9, 1),
                                "frac": round(nbytes_ln / (ms_ln * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
            "l2": "two 235 MB inputs alternated (> 126 MB L2)",
            "timing": f"median of {n} launches each"}


def bench_small(fp8bs, dev, stream, args):
    """The small reference case (M=128, N=256, K=512, FP32 out): quantize A and
    W (one launch) + GEMM per step. A handful of CTAs: launch latency bound,
    so it is reported in microseconds only."""
    d = wl.cfg0(0)
    a = wl.bits_to_torch(d.a_bits).to(dev)
    w = wl.bits_to_torch(d.w_bits).to(dev)
    qa = torch.empty((128, 512), dtype=torch.uint8, device=dev)
    sa = torch.empty((128, 4), dtype=torch.float32, device=dev)
    qw = torch.empty((256, 512), dtype=torch.uint8, device=dev)
    sw = torch.empty((2, 4), dtype=torch.float32, device=dev)
    c = torch.empty((128, 256), dtype=torch.float32, device=dev)

    def step():
        fp8bs.fp8bs_quantize_act_and_weight(a, qa, sa, w, qw, sw, stream)
        fp8bs.fp8bs_gemm(qa, sa, qw, sw, c, stream)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    n = max(20, min(args.steps, 200))
    evs = _events(n)
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            e0.record(stream)
            step()
            e1.record(stream)
    stream.synchronize()
    eager = c.clone()
    # The same step captured once in a CUDA graph and replayed: the host's
    # launch overhead (argument checks, tensor-map encoding, two launches)
    # leaves the timed region.
    graph = {}
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        c.zero_()
        g.replay()
        stream.synchronize()
        gevs = _events(n)
        with torch.cuda.stream(stream):
            for e0, e1 in gevs:
                e0.record(stream)
                g.replay()
                e1.record(stream)
        stream.synchronize()
        graph = {"us_per_step": round(_median_ms(gevs) * 1e3, 2), "same_output": bool(torch.equal(c, eager))}
    except Exception as exc:   # report, do not fail the bench line
        graph = {"error": str(exc)[:200]}
    return {"workload": "quantize + GEMM M=128, N=256, K=512, fp32 out (reference case)",
            "us_per_step": round(_median_ms(evs) * 1e3, 2), "launches_per_step": 2,
            "cuda_graph": graph,
            "timing": f"median of {n} steps (CUDA events); launch-latency bound"}


def bench_gemm2(fp8bs, dev, stream, peaks, args):
    """GEMM M=4096, N=7168, K=2048 (0.5% outlier channels x50), pre-quantized
    operands, bf16 out; operands of 3 seeded sets rotated. Timed beside it:
    the same GEMM preceded by the quantization of both bf16 operands (one
    launch), as a step does."""
    qs, raw = [], []
    for seed in range(3):
        d = wl.cfg2(seed)
        a = wl.bits_to_torch(d.a_bits).to(dev)
        w = wl.bits_to_torch(d.w_bits).to(dev)
        qa, sa = fp8bs.quantize_act(a, stream)
        qw, sw = fp8bs.quantize_weight(w, stream)
        qs.append((qa, sa, qw, sw))
        raw.append((a, w))
    M, K = qs[0][0].shape
    N = qs[0][2].shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = fp8bs.workspace(M, N, K, device=dev)
    n = max(20, min(args.steps, 200))

    def timed(body):
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup)):
                body(i)
        evs = _events(n)
        with torch.cuda.stream(stream):
            for i, (e0, e1) in enumerate(evs):
                e0.record(stream)
                body(i)
                e1.record(stream)
        stream.synchronize()
        assert fp8bs.fp8bs_last_device_error(stream) == fp8bs.OK
        return _median_ms(evs)

    def gemm(i):
        fp8bs.fp8bs_gemm_ws(*qs[i % 3], c, ws, stream)

    def quantize_and_gemm(i):
        qa, sa, qw, sw = qs[i % 3]
        a, w = raw[i % 3]
        fp8bs.fp8bs_quantize_act_and_weight(a, qa, sa, w, qw, sw, stream)
        fp8bs.fp8bs_gemm_ws(qa, sa, qw, sw, c, ws, stream)
    ms = timed(gemm)
    ms_step = timed(quantize_and_gemm)
    flops = 2.0 * M * N * K
    tf = flops / (ms * 1e-3) / 1e12
    fp8_peak = _fp8_peak(peaks)
    return {"workload": "GEMM M=4096,N=7168,K=2048, 0.5% outlier channels x50, bf16 out",
            "us": round(ms * 1e3, 2), "TFLOP/s": round(tf, 1),
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": round(fp8_peak, 1),
                         "unit": "TFLOP/s", "frac": round(tf / fp8_peak, 4),
                         "frac_of_nominal_4500": round(tf / 4500.0, 4)},
            "with_quantize": {"us": round(ms_step * 1e3, 2),
                              "TFLOP/s": round(flops / (ms_step * 1e-3) / 1e12, 1),
                              "launches": 2},
            "timing": f"median of {n} launches (or launch pairs), 3 operand sets rotated"}


def bench_moe(fp8bs, dev, stream, peaks, args, n_tokens=wl.N_TOKENS):
    """Grouped GEMM, 32 experts N=4096 K=7168, pre-quantized operands; rows
    per expert from the seeded top-8 router over n_tokens tokens (8192: the
    prefill/training workload; 256: a decode batch, weight-streaming bound)."""
    counts = wl.moe_routing(0, n_tokens=n_tokens)
    d = wl.moe(seed=0, counts=counts, with_w=False)
    E, N, K = len(d.counts), d.N, d.K
    rng_w = torch.Generator(device=dev)
    rng_w.manual_seed(0)
    # Expert weights: finite E4M3 codes and positive scales drawn on the device
    # from a seeded generator (the kernel's time does not depend on the values).
    qw = torch.randint(0, 0x7F, (E, N, K), dtype=torch.uint8, device=dev, generator=rng_w)
    sw = torch.rand((E, N // 128, K // 128), device=dev, generator=rng_w) * 1e-4
    x = wl.bits_to_torch(d.a_bits).to(dev)
    qa, sa = fp8bs.quantize_act(x, stream)
    off = torch.from_numpy(d.offsets).to(dev)
    total = int(d.offsets[-1])
    c = torch.empty((total, N), dtype=torch.bfloat16, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            fp8bs.fp8bs_grouped_gemm(qa, sa, off, qw, sw, c, stream)
    n = max(10, min(args.steps, 100))
    evs = _events(n)
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            e0.record(stream)
            fp8bs.fp8bs_grouped_gemm(qa, sa, off, qw, sw, c, stream)
            e1.record(stream)
    stream.synchronize()
    assert fp8bs.fp8bs_last_device_error(stream) == fp8bs.OK
    ms = _median_ms(evs)
    flops = 2.0 * total * N * K
    tflops = flops / (ms * 1e-3) / 1e12
    # Algorithmic bytes: every expert's FP8 weights and scales once, the
    # FP8 rows and their scales, the bf16 output.
    wbytes = E * N * K + E * (N // 128) * (K // 128) * 4
    abytes = total * K + total * (K // 128) * 4 + total * N * 2
    fp8_peak = _fp8_peak(peaks)
    t_tensor = flops / (fp8_peak * 1e12)
    t_hbm = (wbytes + abytes) / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    return {"workload": f"MoE grouped GEMM 32 experts N=4096 K=7168, {n_tokens} tokens top-8 over "
                        f"256 experts: rows {total} (max {int(d.counts.max())}, "
                        f"min {int(d.counts.min())})",
            "us": round(ms * 1e3, 2), "TFLOP/s": round(tflops, 1),
            "GB/s": round((wbytes + abytes) / (ms * 1e-3) / 1e9, 1),
            "roofline": {"bound": bound, "achieved_us": round(ms * 1e3, 2),
                         "bound_us": round(max(t_tensor, t_hbm) * 1e6, 2),
                         "frac": round(max(t_tensor, t_hbm) * 1e3 / ms, 4),
                         "tensor_frac": round(tflops / fp8_peak, 4),
                         "hbm_frac": round((wbytes + abytes) / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
            "timing": f"median of {n} launches; weights 940 MB > L2"}


def bench_e2e(fp8bs, dev, stream, args, world=1):
    """Same step through the C entry points from pinned host buffers: every
    step copies A and W (bf16) host -> device, quantizes both (one launch),
    runs the GEMM and copies C device -> host. Uploads run on their own
    stream into alternating device buffers, so step i+1's uploads overlap
    step i's kernels; C's copy back runs on a third stream (C alternates
    between two buffers too)."""
    d = wl.cfg3(seed=0)
    a_h = wl.bits_to_torch(d.a_bits).pin_memory()
    w_h = wl.bits_to_torch(d.w_bits).pin_memory()
    c_h = [torch.empty((M3, N3), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    a = [torch.empty((M3, K3), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    w = [torch.empty((N3, K3), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    qa = torch.empty((M3, K3), dtype=torch.uint8, device=dev)
    sa = torch.empty((M3, K3 // 128), dtype=torch.float32, device=dev)
    qw = torch.empty((N3, K3), dtype=torch.uint8, device=dev)
    sw = torch.empty((N3 // 128, K3 // 128), dtype=torch.float32, device=dev)
    c = [torch.empty((M3, N3), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws = fp8bs.workspace(M3, N3, K3, device=dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]
    gemm_done = [torch.cuda.Event(), torch.cuda.Event()]
    out_done = [torch.cuda.Event(), torch.cuda.Event()]

    def step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(consumed[b])       # step i-2's quantizer has read a[b], w[b]
            a[b].copy_(a_h, non_blocking=True)
            w[b].copy_(w_h, non_blocking=True)
            in_ready[b].record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready[b])
            stream.wait_event(out_done[b])     # step i-2's copy-out of C[b] is done
            fp8bs.fp8bs_quantize_act_and_weight(a[b], qa, sa, w[b], qw, sw, stream)
            consumed[b].record(stream)
            fp8bs.fp8bs_gemm_ws(qa, sa, qw, sw, c[b], ws, stream)
            gemm_done[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(gemm_done[b])
            c_h[b].copy_(c[b], non_blocking=True)
            out_done[b].record(s_out)

    def drain():
        stream.wait_event(out_done[0])
        stream.wait_event(out_done[1])
        stream.wait_event(in_ready[0])
        stream.wait_event(in_ready[1])

    for i in range(max(3, args.warmup)):
        step(i)
    drain()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    n = max(10, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(n):
        step(i)
    drain()
    e1.record(stream)
    stream.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / n
    flops = 2.0 * M3 * N3 * K3
    return {"value": round(world * flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": world * 2 * (M3 * K3 + N3 * K3), "d2h_bytes_per_step": world * 2 * M3 * N3,
            "ms_per_step": round(ms, 4), "steps": n,
            "path": "pinned host A, W -> H2D (upload stream, alternating buffers) -> quantize A + W "
                    "(one launch), GEMM -> D2H C (third stream); uploads and copy-back overlap "
                    "the kernels of neighbouring steps"}


def run_ours(args, world):
    from fp8_fine_grained_17_b300 import fp8bs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    peaks = _peaks()
    parts = {"all": ("step", "small", "act_quant", "norm_quant", "fused", "gemm2", "moe", "e2e"),
             "replicas": ("step", "e2e")}.get(args.part, (args.part,))

    result = {}
    if "step" in parts:
        s = bench_step(fp8bs, dev, stream, peaks, args, world)
        result = {
            "metric": METRIC, "value": round(s["value"], 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(s["elapsed_ms"] / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic (seeded numpy N(0,1) activations, N(0,0.02) weights, bf16)",
            "config": line_config(world),
            "method": {"kernel_events": f"per-kernel CUDA events on every {EVENT_EVERY}th timed step",
                       "launch": "the GEMM is launched as a programmatic dependent of the quantizer",
                       "input_sets": f"{s['n_sets']} seeded sets, {s['set_bytes'] / 1e6:.0f} MB"},
            "roofline": s["roofline"],
            "kernels": s["kernels"],
            "gpu_launches": 2 * args.steps,
            "clocks": s["clocks"],
        }
        torch.cuda.empty_cache()
    if "small" in parts:
        result["small_reference_case"] = bench_small(fp8bs, dev, stream, args)
    if "act_quant" in parts:
        result["act_quant"] = bench_act_quant(fp8bs, dev, stream, peaks, args)
        torch.cuda.empty_cache()
    if "norm_quant" in parts:
        result["norm_quant"] = bench_norm_quant(fp8bs, dev, stream, peaks, args)
        torch.cuda.empty_cache()
    if "fused" in parts:
        result["fused_act_quant_gemm"] = bench_fused(fp8bs, dev, stream, peaks, args)
        torch.cuda.empty_cache()
    if "gemm2" in parts:
        result["gemm_4096x7168x2048"] = bench_gemm2(fp8bs, dev, stream, peaks, args)
        torch.cuda.empty_cache()
    if "moe" in parts:
        result["moe_grouped"] = bench_moe(fp8bs, dev, stream, peaks, args)
        torch.cuda.empty_cache()
        result["moe_decode"] = bench_moe(fp8bs, dev, stream, peaks, args, n_tokens=256)
        torch.cuda.empty_cache()
    if "e2e" in parts:
        result["e2e"] = bench_e2e(fp8bs, dev, stream, args, world)
    return result


# --------------------------------------------------------------- oracle (CPU)

def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d["num_threads"] for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def _oracle_step(orc, a_bits, w_bits):
    qa, sa = orc.quantize_act_1x128(a_bits)
    qw, sw = orc.quantize_weight_128x128(w_bits)
    orc.gemm(qa, sa, qw, sw)


def _oracle_sample(orc, budget_s: float):
    """Rows of A for one oracle step of about budget_s seconds: the step is
    quantize A[rows, 7168] + quantize W[4096, 7168] + float64 GEMM
    rows x 4096 x 7168, so its time is affine in rows; fit it from two runs."""
    d = wl.cfg3(seed=0)
    ts = []
    for r in (8, 32):
        t = time.perf_counter()
        _oracle_step(orc, d.a_bits[:r], d.w_bits)
        ts.append(time.perf_counter() - t)
    per_row = max((ts[1] - ts[0]) / 24, 1e-6)
    fixed = max(ts[0] - 8 * per_row, 0.0)
    rows = int(np.clip((budget_s - fixed) / per_row, 8, M3))
    return d, rows


def cpu_baseline(budget_s: float = 15.0):
    """The oracle (C quantizers + float64 numpy GEMM) on a bounded sample of
    the step: the first `rows` rows of A with all of W, i.e. a rows x 4096 x
    7168 slice of the same GEMM (all 4096 rows when that fits the budget);
    TFLOP/s counts the sample's own FLOPs."""
    from oracle import oracle as orc
    with _all_host_cores():
        d, rows = _oracle_sample(orc, budget_s)
        rows = M3 if rows >= M3 // 4 else rows
        t = time.perf_counter()
        _oracle_step(orc, d.a_bits[:rows], d.w_bits)
        dt = time.perf_counter() - t
        cores = _blas_threads()
    flops = 2.0 * rows * N3 * K3
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"quantize A[{rows},{K3}] + W[{N3},{K3}] (plain C, 1 thread) and float64 "
                      f"GEMM {rows}x{N3}x{K3} (numpy BLAS, {cores} threads) in {dt:.2f} s",
            "seconds": round(dt, 2)}


def _all_host_cores():
    """BLAS on every host core for the oracle (torchrun sets OMP_NUM_THREADS=1
    for each rank; under torchrun only rank 0 runs the oracle)."""
    try:
        from threadpoolctl import threadpool_limits
        return threadpool_limits(limits=os.cpu_count() or 1, user_api="blas")
    except Exception:
        import contextlib
        return contextlib.nullcontext()


def run_reference(args, world: int = 1):
    """The oracle timed on the host cores: W + K steps, each a bounded sample
    (rows x 4096 x 7168 slice) of the headline step. Under torchrun rank 0
    alone runs it."""
    from oracle import oracle as orc
    per_step = float(np.clip(150.0 / max(1, args.steps + args.warmup), 0.5, 15.0))
    with _all_host_cores():
        d, rows = _oracle_sample(orc, per_step)
        for _ in range(args.warmup):
            _oracle_step(orc, d.a_bits[:rows], d.w_bits)
        t = time.perf_counter()
        for _ in range(args.steps):
            _oracle_step(orc, d.a_bits[:rows], d.w_bits)
        dt = time.perf_counter() - t
        cores = _blas_threads()
    flops = 2.0 * rows * N3 * K3
    value = flops * args.steps / dt / 1e12
    sample = (f"per step: quantize A[{rows},{K3}] + W[{N3},{K3}] (plain C, 1 thread) + float64 "
              f"GEMM {rows}x{N3}x{K3} (numpy BLAS, {cores} threads)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(world),
            "method": {"sample_rows": rows,
                       "ranks": "rank 0 runs the oracle on the host; other ranks exit"
                                if world > 1 else "one process on the host"},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--part", choices=["all", "step", "small", "act_quant", "norm_quant", "fused", "gemm2",
                                       "moe", "e2e"],
                    default="all", help="which measurements to run (profiling uses one)")
    ap.add_argument("--skip-cpu", action="store_true", help="no oracle CPU baseline")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
        if args.part == "all":
            args.part = "replicas"   # the step and e2e; the extras are single-GPU measurements
    res = run_ours(args, world)
    if rank == 0:
        if world == 1 and not args.skip_cpu and args.part == "all":
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
