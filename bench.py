#!/usr/bin/env python3
"""Benchmark of the fine-grained FP8 GEMM path on B300.

One step = one FP8 forward of a linear layer at M=4096, N=4096, K=7168 from
bf16 inputs: activation quantization (1x128 tiles), weight quantization
(128x128 blocks), and the block-scaled GEMM with bf16 output. The headline
value is GEMM TFLOP/s over the whole step. The same run also measures the
activation quantizer alone on [16384, 7168] (GB/s) and the MoE grouped GEMM
(32 experts, N=4096, K=7168, seeded top-8 routing) as extra keys.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (launched by torchrun) every rank runs the same step on its
own GPU with no collective on the data path (independent replicas, weak
scaling); the value is the sum of all ranks' work over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_fine_grained_17_b300 import workloads as wl  # noqa: E402

L2_BYTES = 126 * 2 ** 20
METRIC = "FP8 block-scaled GEMM TFLOP/s (% of dense FP8 peak); act-quant HBM GB/s"
UNIT = "TFLOP/s"
WORKLOAD = "GEMM M=4096,N=4096,K=7168: A bf16 ~N(0,1), W bf16 ~N(0,0.02), block-quantized to E4M3, bf16 out"
M3, N3, K3 = 4096, 4096, 7168


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML while running."""

    REASONS = {
        "sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
    }

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._period = period_s
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nvml = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
        except Exception:
            self._nvml = None
        self._t = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self._nvml.nvmlDeviceGetClockInfo(self._h, self._nvml.NVML_CLOCK_SM))
                r = self._nvml.nvmlDeviceGetCurrentClocksEventReasons(self._h)
                for name, bit in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self._period)

    def __enter__(self):
        if self._nvml is not None:
            self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._nvml is not None:
            self._t.join()

    def summary(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples), "source": "nvml"}


# --------------------------------------------------------------------- our arm

def _dense_inputs(n_sets: int, dev):
    """n_sets independent seeded (A, W) bf16 pairs on the device."""
    sets = []
    for i in range(n_sets):
        d = wl.cfg3(seed=i)
        sets.append((wl.bits_to_torch(d.a_bits).to(dev), wl.bits_to_torch(d.w_bits).to(dev)))
    return sets


def run_ours(args, rank, world):
    from fp8_fine_grained_17_b300 import fp8bs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    peaks = _peaks()

    step_in_bytes = 2 * (M3 * K3 + N3 * K3)
    n_sets = max(2, -(-3 * L2_BYTES // step_in_bytes))
    sets = _dense_inputs(n_sets, dev)
    qa = torch.empty((M3, K3), dtype=torch.uint8, device=dev)
    sa = torch.empty((M3, K3 // 128), dtype=torch.float32, device=dev)
    qw = torch.empty((N3, K3), dtype=torch.uint8, device=dev)
    sw = torch.empty((N3 // 128, K3 // 128), dtype=torch.float32, device=dev)
    c = torch.empty((M3, N3), dtype=torch.bfloat16, device=dev)

    def step(i, ev=None):
        a, w = sets[i % n_sets]
        if ev is not None:
            ev[0].record(stream)
        fp8bs.fp8bs_quantize_act_1x128(a, qa, sa, stream)
        if ev is not None:
            ev[1].record(stream)
        fp8bs.fp8bs_quantize_weight_128x128(w, qw, sw, stream)
        if ev is not None:
            ev[2].record(stream)
        fp8bs.fp8bs_gemm(qa, sa, qw, sw, c, stream)
        if ev is not None:
            ev[3].record(stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(args.steps):
                step(i, evs[i])
            t1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    elapsed_ms = t0.elapsed_time(t1)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        elapsed_ms = float(t.item())
        torch.distributed.barrier()
    assert fp8bs.fp8bs_last_device_error(stream) == fp8bs.OK

    per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])]
                    for e in evs])
    t_qa, t_qw, t_gemm = per.mean(axis=0)
    flops = 2.0 * M3 * N3 * K3
    ms_per_step = elapsed_ms / args.steps
    value = world * flops * args.steps / (elapsed_ms * 1e-3) / 1e12
    fp8_peak = peaks["bf16_tflops"] * 2.0      # measured bf16 burst x nominal fp8/bf16 ratio (4.5/2.25)
    gemm_tflops = flops / (t_gemm * 1e-3) / 1e12
    qa_bytes = M3 * K3 * 2 + M3 * K3 + M3 * (K3 // 128) * 4
    qw_bytes = N3 * K3 * 2 + N3 * K3 + (N3 // 128) * (K3 // 128) * 4

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded numpy N(0,1) activations, N(0,0.02) weights, bf16)",
        "config": {"workload": WORKLOAD, "M": M3, "N": N3, "K": K3, "out": "bf16",
                   "step": "quantize A 1x128 + quantize W 128x128 + block-scaled GEMM",
                   "l2": f"inputs rotated over {n_sets} seeded sets "
                         f"({n_sets * step_in_bytes / 1e6:.0f} MB > 126 MB L2), no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "fp8_gemm_kernel",
                     "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4),
                     "traffic": None,
                     "peak_note": f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} x 2 (nominal fp8/bf16)",
                     "frac_of_nominal_4500": round(gemm_tflops / 4500.0, 4)},
        "kernels": {
            "quantize_act_1x128": {"ms": round(t_qa, 4), "GB/s": round(qa_bytes / (t_qa * 1e-3) / 1e9, 1),
                                   "frac_hbm": round(qa_bytes / (t_qa * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
            "quantize_weight_128x128": {"ms": round(t_qw, 4), "GB/s": round(qw_bytes / (t_qw * 1e-3) / 1e9, 1),
                                        "frac_hbm": round(qw_bytes / (t_qw * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
            "gemm": {"ms": round(t_gemm, 4), "TFLOP/s": round(gemm_tflops, 1)},
        },
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
    }
    del sets
    torch.cuda.empty_cache()
    if not args.skip_extras:
        result["act_quant"] = bench_act_quant(fp8bs, dev, stream, peaks, args)
        result["moe_grouped"] = bench_moe(fp8bs, dev, stream, peaks, args)
        result["e2e"] = bench_e2e(fp8bs, dev, stream, args)
    return result


def bench_act_quant(fp8bs, dev, stream, peaks, args):
    """Activation quantizer alone on [16384, 7168] with 0.5% outlier channels x100."""
    d = wl.cfg1(0)
    x = wl.bits_to_torch(d.a_bits).to(dev)
    M, K = x.shape
    q = torch.empty((M, K), dtype=torch.uint8, device=dev)
    s = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            fp8bs.fp8bs_quantize_act_1x128(x, q, s, stream)
    n = max(20, args.steps)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            e0.record(stream)
            fp8bs.fp8bs_quantize_act_1x128(x, q, s, stream)
            e1.record(stream)
    stream.synchronize()
    ms = float(np.median([a.elapsed_time(b) for a, b in evs]))
    nbytes = M * K * 2 + M * K + M * (K // 128) * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "act-quant [16384,7168] bf16, 36 outlier channels x100", "ms": round(ms, 4),
            "GB/s": round(gbs, 1), "bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "frac_of_8000": round(gbs / 8000.0, 4)},
            "l2": "input 235 MB > 126 MB L2", "timing": f"median of {n} launches"}


def bench_moe(fp8bs, dev, stream, peaks, args):
    """Grouped GEMM, 32 experts N=4096 K=7168, pre-quantized operands."""
    d = wl.moe(seed=0, with_w=False)
    E, N, K = len(d.counts), d.N, d.K
    rng_w = torch.Generator(device=dev)
    rng_w.manual_seed(0)
    # Expert weights: codes and scales drawn on the device from a seeded
    # generator (the kernel's time does not depend on the values).
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
    n = max(10, args.steps // 2)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            e0.record(stream)
            fp8bs.fp8bs_grouped_gemm(qa, sa, off, qw, sw, c, stream)
            e1.record(stream)
    stream.synchronize()
    assert fp8bs.fp8bs_last_device_error(stream) == fp8bs.OK
    ms = float(np.median([a.elapsed_time(b) for a, b in evs]))
    flops = 2.0 * total * N * K
    tflops = flops / (ms * 1e-3) / 1e12
    wbytes = E * N * K
    fp8_peak = peaks["bf16_tflops"] * 2.0
    t_bound = max(flops / (fp8_peak * 1e12), wbytes / (peaks["hbm_gbs"] * 1e9))
    return {"workload": f"MoE grouped GEMM 32 experts N=4096 K=7168, rows {total} "
                        f"(max {int(d.counts.max())}, min {int(d.counts.min())})",
            "ms": round(ms, 4), "TFLOP/s": round(tflops, 1), "weight_bytes": wbytes,
            "roofline": {"bound": "tensor+weight stream", "achieved_ms": round(ms, 4),
                         "bound_ms": round(t_bound * 1e3, 4), "frac": round(t_bound * 1e3 / ms, 4),
                         "tensor_frac": round(tflops / fp8_peak, 4)},
            "timing": f"median of {n} launches; weights 940 MB > L2"}


def bench_e2e(fp8bs, dev, stream, args):
    """Same step through the C entry points from pinned host buffers: H2D of
    A and W (bf16), quantize, quantize, GEMM, D2H of C, every step."""
    d = wl.cfg3(seed=0)
    a_h = wl.bits_to_torch(d.a_bits).pin_memory()
    w_h = wl.bits_to_torch(d.w_bits).pin_memory()
    c_h = torch.empty((M3, N3), dtype=torch.bfloat16).pin_memory()
    a = torch.empty((M3, K3), dtype=torch.bfloat16, device=dev)
    w = torch.empty((N3, K3), dtype=torch.bfloat16, device=dev)
    qa = torch.empty((M3, K3), dtype=torch.uint8, device=dev)
    sa = torch.empty((M3, K3 // 128), dtype=torch.float32, device=dev)
    qw = torch.empty((N3, K3), dtype=torch.uint8, device=dev)
    sw = torch.empty((N3 // 128, K3 // 128), dtype=torch.float32, device=dev)
    c = torch.empty((M3, N3), dtype=torch.bfloat16, device=dev)

    def step():
        a.copy_(a_h, non_blocking=True)
        w.copy_(w_h, non_blocking=True)
        fp8bs.fp8bs_quantize_act_1x128(a, qa, sa, stream)
        fp8bs.fp8bs_quantize_weight_128x128(w, qw, sw, stream)
        fp8bs.fp8bs_gemm(qa, sa, qw, sw, c, stream)
        c_h.copy_(c, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
        stream.synchronize()
        n = max(10, args.steps // 2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            step()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / n
    flops = 2.0 * M3 * N3 * K3
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": 2 * (M3 * K3 + N3 * K3), "d2h_bytes_per_step": 2 * M3 * N3,
            "ms_per_step": round(ms, 4), "steps": n}


# --------------------------------------------------------------- oracle (CPU)

def _oracle_step(orc, a_bits, w_bits):
    qa, sa = orc.quantize_act_1x128(a_bits)
    qw, sw = orc.quantize_weight_128x128(w_bits)
    orc.gemm(qa, sa, qw, sw)


def cpu_baseline(budget_s: float = 15.0, rows: int | None = None):
    """The oracle (C quantizers + float64 numpy GEMM) on a bounded sample of
    the step: the first `rows` rows of A and the first rows of W, so the
    sample is (rows x 4096-column-slice) of the same GEMM; TFLOP/s scaled by
    the sample's own FLOPs."""
    from oracle import oracle as orc
    d = wl.dense("sample", 256, N3, K3, seed=0)
    a_bits, w_bits = d.a_bits, d.w_bits
    # calibrate on a small slice
    t = time.perf_counter()
    _oracle_step(orc, a_bits[:16], w_bits[:256])
    t_small = time.perf_counter() - t
    if rows is None:
        rows = int(np.clip(16 * budget_s / max(t_small, 1e-3) / 16, 16, 256))
    n_cols = 256 * max(1, min(N3 // 256, int(budget_s / max(t_small, 1e-3))))
    t = time.perf_counter()
    _oracle_step(orc, a_bits[:rows], w_bits[:n_cols])
    dt = time.perf_counter() - t
    flops = 2.0 * rows * n_cols * K3
    threads = int(os.environ.get("OMP_NUM_THREADS", 0)) or os.cpu_count()
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"quantize A[{rows},{K3}] + W[{n_cols},{K3}] (C, 1 thread) and float64 GEMM "
                      f"{rows}x{n_cols}x{K3} (numpy BLAS) in {dt:.2f} s",
            "seconds": round(dt, 2)}


def run_reference(args, rank):
    """The oracle timed on the host cores, K timed steps of a bounded sample."""
    from oracle import oracle as orc
    d = wl.dense("sample", 64, N3, K3, seed=0)
    budget_per_step = max(0.2, 150.0 / max(1, args.steps + args.warmup))
    t = time.perf_counter()
    _oracle_step(orc, d.a_bits[:8], d.w_bits[:256])
    t_small = time.perf_counter() - t
    scale = max(1.0, budget_per_step / max(t_small, 1e-3))
    rows = int(min(64, 8 * scale ** 0.5))
    n_cols = int(min(N3, 256 * max(1, int(scale ** 0.5))) // 256 * 256)
    for _ in range(args.warmup):
        _oracle_step(orc, d.a_bits[:rows], d.w_bits[:n_cols])
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(orc, d.a_bits[:rows], d.w_bits[:n_cols])
    dt = time.perf_counter() - t
    flops = 2.0 * rows * n_cols * K3
    value = flops * args.steps / dt / 1e12
    cores = int(os.environ.get("OMP_NUM_THREADS", 0)) or os.cpu_count()
    sample = f"quantize A[{rows},{K3}] + W[{n_cols},{K3}] + float64 GEMM {rows}x{n_cols}x{K3} per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "M": M3, "N": N3, "K": K3},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-extras", action="store_true", help="headline step only")
    ap.add_argument("--skip-cpu", action="store_true", help="no oracle CPU baseline")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        if world == 1 and not args.skip_cpu:
            res["cpu_baseline"] = cpu_baseline()
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
