"""Shared test helpers: move seeded inputs to the GPU, run the library through
its C entry points, and compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

from fp8_fine_grained_17_b300 import fp8bs
from fp8_fine_grained_17_b300 import workloads as wl


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return wl.bits_to_torch(bits).cuda()


def gpu_quant_act(bits: np.ndarray):
    x = to_dev_bf16(bits)
    q, s = fp8bs.quantize_act(x)
    return q, s


def gpu_quant_weight(bits: np.ndarray):
    w = to_dev_bf16(bits)
    q, s = fp8bs.quantize_weight(w)
    return q, s


def check_codes(q_gpu: torch.Tensor, s_gpu: torch.Tensor, q_or: np.ndarray, s_or: np.ndarray):
    qg = q_gpu.cpu().numpy()
    sg = s_gpu.cpu().numpy()
    bad_s = np.flatnonzero(sg.view(np.uint32).ravel() != s_or.view(np.uint32).ravel())
    assert bad_s.size == 0, f"{bad_s.size} scales differ, first at {bad_s[:5]}"
    bad_q = np.flatnonzero(qg.ravel() != q_or.ravel())
    assert bad_q.size == 0, (f"{bad_q.size} codes differ, first at {bad_q[:5]}: "
                             f"gpu {qg.ravel()[bad_q[:5]]} oracle {q_or.ravel()[bad_q[:5]]}")


def check_gemm(c_gpu: torch.Tensor, C_or: np.ndarray, B: np.ndarray, out_bf16: bool):
    got = c_gpu.float().cpu().numpy().astype(np.float64)
    tol = 2e-5 * B + 1e-6
    if out_bf16:
        tol = tol + np.abs(C_or) * 2.0 ** -8
    err = np.abs(got - C_or)
    bad = np.flatnonzero((err > tol).ravel())
    worst = float(np.max(err / tol)) if err.size else 0.0
    assert bad.size == 0, (f"{bad.size}/{err.size} outside tolerance; worst err/tol {worst:.3g}; "
                           f"first {bad[:5]} got {got.ravel()[bad[:5]]} want {C_or.ravel()[bad[:5]]}")
    return worst
