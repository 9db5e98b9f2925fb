"""Seeded synthetic inputs for the fine-grained FP8 path.

This module only draws random numbers and rounds them to bf16 input tensors;
it holds none of the method's arithmetic. Both the CUDA path's tests and
benchmark and the CPU oracle's checks take their inputs from here.

Recipes (numpy ``default_rng``; fp32 draws rounded to bf16 with
round-to-nearest-even):

* ``dense(...)``: A ~ N(0, 1) of shape [M, K]; optionally a seeded 0.5% of the
  K channels (``round(0.005 K)`` columns chosen without replacement) scaled by
  an outlier factor before rounding; W ~ N(0, 0.02^2) of shape [N, K].
* ``moe_routing(...)``: 8192 tokens routed top-8 over 256 experts. Expert
  popularity follows Zipf weights p_r ~ r^-1.1 over ranks r = 1..256, the
  rank of each expert given by a seeded permutation; each token takes 8
  distinct experts drawn without replacement in proportion to p (Gumbel
  top-8). The local experts are ids 0..31 and the rows of local expert e
  are the tokens that chose it.
* ``moe(...)``: the routing above, W_e ~ N(0, 0.02^2) of shape [32, N, K],
  and A ~ N(0, 1) of shape [sum_e M_e, K] with rows sorted by expert.

The pages measure on no public dataset, so these synthetic tensors stand in
for the activations and weights of the model layers they describe (MoE with
256 routed experts, top-8, expert hidden 2048: "How I Improved My Deepseek
In In The Future", paragraph on the MoE layer).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

OUTLIER_FRACTION = 0.005


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); uint16 patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact float32 values of bf16 patterns."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bits_to_torch(b: np.ndarray) -> torch.Tensor:
    """bf16 torch tensor (CPU) sharing the patterns in ``b``."""
    return torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def _children(seed: int, n: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(n)]


def activations(rng: np.random.Generator, M: int, K: int, outlier_scale: float | None = None):
    """A ~ N(0,1) [M, K] as bf16 patterns, with optional outlier channels."""
    a = rng.standard_normal((M, K), dtype=np.float32)
    cols = np.zeros(0, dtype=np.int64)
    if outlier_scale is not None:
        n_out = int(round(OUTLIER_FRACTION * K))
        cols = np.sort(rng.choice(K, size=n_out, replace=False))
        a[:, cols] *= np.float32(outlier_scale)
    return bf16_bits(a), cols


def weights(rng: np.random.Generator, N: int, K: int, std: float = 0.02):
    """W ~ N(0, std^2) [N, K] as bf16 patterns."""
    return bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * np.float32(std))


@dataclass
class Dense:
    name: str
    M: int
    N: int
    K: int
    a_bits: np.ndarray | None
    w_bits: np.ndarray | None
    outlier_cols: np.ndarray
    out_bf16: bool


def dense(name: str, M: int, N: int, K: int, seed: int = 0, outlier_scale=None,
          out_bf16: bool = True, with_w: bool = True) -> Dense:
    ra, rw = _children(seed, 2)
    a, cols = activations(ra, M, K, outlier_scale)
    w = weights(rw, N, K) if with_w else None
    return Dense(name, M, N, K, a, w, cols, out_bf16)


# The five workloads of the fine-grained FP8 path.
def cfg0(seed: int = 0) -> Dense:
    """Quantize + GEMM reference case: M=128, N=256, K=512, FP32 output."""
    return dense("quant+gemm M=128 N=256 K=512 f32-out", 128, 256, 512, seed, None, out_bf16=False)


def cfg1(seed: int = 0) -> Dense:
    """Activation quantize only: A [16384, 7168], 0.5% channels x100."""
    return dense("act-quant [16384,7168] outliers x100", 16384, 0, 7168, seed, 100.0, with_w=False)


def cfg2(seed: int = 0) -> Dense:
    """GEMM M=4096, N=7168, K=2048, 0.5% channels x50, bf16 output."""
    return dense("gemm M=4096 N=7168 K=2048 outliers x50 bf16-out", 4096, 7168, 2048, seed, 50.0)


def cfg3(seed: int = 0) -> Dense:
    """GEMM M=4096, N=4096, K=7168, bf16 output."""
    return dense("gemm M=4096 N=4096 K=7168 bf16-out", 4096, 4096, 7168, seed, None)


N_TOKENS = 8192
N_EXPERTS = 256
TOP_K = 8
N_LOCAL = 32
ZIPF_S = 1.1


def moe_routing(seed: int = 0, n_tokens: int = N_TOKENS, n_experts: int = N_EXPERTS,
                top_k: int = TOP_K, n_local: int = N_LOCAL) -> np.ndarray:
    """Rows per local expert (int64 [n_local]) from the seeded top-k router."""
    rng = _children(seed, 3)[0]
    p = np.arange(1, n_experts + 1, dtype=np.float64) ** -ZIPF_S
    p /= p.sum()
    rank = rng.permutation(n_experts)               # expert e has rank rank[e] + 1
    logp = np.log(p[rank])
    counts = np.zeros(n_experts, dtype=np.int64)
    chunk = 1024
    for t0 in range(0, n_tokens, chunk):
        t = min(chunk, n_tokens - t0)
        keys = logp[None, :] + rng.gumbel(size=(t, n_experts))
        chosen = np.argpartition(-keys, top_k - 1, axis=1)[:, :top_k]
        counts += np.bincount(chosen.ravel(), minlength=n_experts)
    return counts[:n_local]


@dataclass
class MoE:
    name: str
    counts: np.ndarray      # rows per local expert
    offsets: np.ndarray     # int32 [E+1]
    N: int
    K: int
    a_bits: np.ndarray | None
    w_bits: np.ndarray | None   # [E, N, K]


def moe(seed: int = 0, N: int = 4096, K: int = 7168, counts=None, with_a: bool = True,
        with_w: bool = True) -> MoE:
    """MoE up-projection: 32 local experts, rows from the router above."""
    _, rw, ra = _children(seed, 3)
    if counts is None:
        counts = moe_routing(seed)
    counts = np.asarray(counts, dtype=np.int64)
    offsets = np.zeros(len(counts) + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    E = len(counts)
    w = None
    if with_w:
        w = np.empty((E, N, K), dtype=np.uint16)
        for e in range(E):
            w[e] = weights(rw, N, K)
    a = activations(ra, int(offsets[-1]), K)[0] if with_a else None
    return MoE(f"moe grouped {E} experts N={N} K={K} rows={int(offsets[-1])}",
               counts, offsets, N, K, a, w)


def norm_params(rng: np.random.Generator, K: int, with_beta: bool):
    """Normalization weights as bf16 patterns: gamma ~ 1 + N(0, 0.1^2) [K] and,
    if asked, beta ~ N(0, 0.02^2) [K]."""
    gamma = bf16_bits(np.float32(1.0) + rng.standard_normal(K, dtype=np.float32) * np.float32(0.1))
    beta = bf16_bits(rng.standard_normal(K, dtype=np.float32) * np.float32(0.02)) if with_beta else None
    return gamma, beta


@dataclass
class Norm:
    name: str
    M: int
    K: int
    x_bits: np.ndarray
    gamma_bits: np.ndarray
    beta_bits: np.ndarray | None


def norm(M: int, K: int, seed: int = 0, outlier_scale=100.0, with_beta: bool = False) -> Norm:
    """Hidden states entering a normalization layer: the activation recipe
    (N(0,1), 0.5% outlier channels) and the weights of ``norm_params``."""
    rx, rp = _children(seed + 1000, 2)
    x, _ = activations(rx, M, K, outlier_scale)
    gamma, beta = norm_params(rp, K, with_beta)
    return Norm(f"norm+quant [{M},{K}]", M, K, x, gamma, beta)
