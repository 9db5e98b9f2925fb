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


U32 = 2.0 ** -24   # unit roundoff of binary32


def norm_rstd_bound(K: int) -> float:
    """Relative bound on |rstd_kernel - rstd_oracle| for rows of K elements.

    The kernel sums each row in binary32 along chains of at most K/64 + 15
    additions (lane-local accumulators, the combination of a lane's
    accumulators, a 5-level butterfly and, for rows split over warps, the warp
    partials), so the sum is off by at most (K/64 + 15) u relative (+2 u for
    LayerNorm's rounded differences). 1/sqrt halves that; the division by K,
    the + eps and the rounded 1/sqrt add 3 u, the oracle's own rounding to
    binary32 one more."""
    return ((K / 64 + 15) / 2 + 4) * U32


def norm_mu_bound(x_bits: np.ndarray, mu_or: np.ndarray) -> np.ndarray:
    """Absolute bound on |mu_kernel - mu_oracle| per row (LayerNorm): the sum's
    chain error (K/64 + 16) u sum|x|, the division and the oracle's rounding."""
    K = x_bits.shape[1]
    mag = np.abs(wl.bits_to_f32(x_bits).astype(np.float64)).mean(axis=1)
    return (K / 64 + 16) * U32 * mag + 2 * U32 * np.abs(mu_or.astype(np.float64))


def check_norm_rows(orc, x_bits, g_bits, b_bits, kind, eps, q, s, mean_k, rstd_k, max_ring=64):
    """Fused normalization + 1x128 cast against the oracle.

    (1) The kernel's row statistics lie inside the proven intervals around
    the oracle's own (correctly rounded) statistics. (2) Every row of codes
    and scales equals the oracle's row at some binary32 statistic inside those
    intervals; the oracle enumerates the candidates from its own statistics
    outward (nothing from the kernel enters it) and the first match counts.
    Returns (rows compared, rows that needed a non-central statistic, the
    farthest ring used)."""
    q = q.cpu().numpy() if torch.is_tensor(q) else np.asarray(q)
    s = s.cpu().numpy() if torch.is_tensor(s) else np.asarray(s)
    M, K = x_bits.shape
    mu_or, r_or = orc.norm_stats(x_bits, kind, eps)
    r_rel = norm_rstd_bound(K)
    rel = np.abs(np.asarray(rstd_k, np.float64) - r_or) / r_or
    assert rel.max() <= r_rel, f"rstd off by {rel.max() / U32:.1f} u (bound {r_rel / U32:.1f} u)"
    mu_abs = np.zeros(M)
    if kind == orc.NORM_LAYER:
        mu_abs = norm_mu_bound(x_bits, mu_or)
        err = np.abs(np.asarray(mean_k, np.float64) - mu_or)
        assert np.all(err <= mu_abs), f"mean off by {np.max(err / np.maximum(mu_abs, 1e-300)):.3g} x bound"
    q_c, s_c, _, _, _ = orc.norm_quantize_act_1x128(x_bits, g_bits, b_bits, kind, eps)
    s_u = s.view(np.uint32)
    same = np.all(q == q_c, axis=1) & np.all(s_u == s_c.view(np.uint32), axis=1)
    rings = []
    for i in np.flatnonzero(~same):
        found = None
        for d, mus, rs in orc.norm_stat_rings(mu_or[i], r_or[i], kind, mu_abs[i], r_rel, max_ring):
            if d == 0:
                continue
            qc, sc = orc.norm_rows_at(x_bits[i], g_bits, b_bits, kind, mus, rs)
            hit = np.all(qc == q[i], axis=1) & np.all(sc.view(np.uint32) == s_u[i], axis=1)
            if hit.any():
                found = d
                break
        assert found is not None, (
            f"row {i}: no admissible statistic within {max_ring} ulps reproduces the kernel's row "
            f"({int(np.sum(q[i] != q_c[i]))} codes, {int(np.sum(s_u[i] != s_c[i].view(np.uint32)))} scales "
            f"differ from the central row)")
        rings.append(found)
    return M, len(rings), max(rings, default=0)
