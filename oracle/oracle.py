"""CPU oracle for the fine-grained FP8 GEMM path.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The product path
(the CUDA library ``libfp8bs.so`` and its Python binding) never does; the two
share no code.

What it computes, and the passage each step follows:

* FP8 encoding and the two quantizers live in ``fp8bs_oracle.c`` (plain C,
  binary32 arithmetic as the statement of the problem fixes it: s = amax/448,
  q = RNE-saturate(x/s) to E4M3). Grouping per 1x128 activation tile and per
  128x128 weight block: "personal notes concerning the deepseek core
  readings" (why-be.why-be.co.kr), fine-grained quantization paragraph,
  Figure 7(a).
* The GEMM is the plain definition the method approximates: dequantize both
  operands exactly in float64 (code value times its group's scale) and
  contract over K, C = A_hat @ W_hat^T. The pages apply the per-group scales
  along K during dequantization with FP32 accumulation on CUDA cores
  (Q&A post on xn--9g3bo1gtkw0l8ubf92bgle.kr, paragraph on per-group scaling
  factors along the inner dimension K; "How Google Is Changing How We Method
  Deepseek", paragraph on limited accumulation bit width); up to rounding
  order that is exactly this contraction. The matmul is numpy's float64
  routine, used as a library primitive.
* Grouped (MoE) GEMM: the same contraction per expert slice of rows (Q&A
  post, paragraph on quantizing before the MoE up-projection for FP8 Fprop).
* Acceptance bound: |C_gpu - C_or| <= 2e-5 * sum_k |A_hat W_hat| + 1e-6, plus
  2^-8 |C_or| for a bf16 output (statement of the problem).
* Power-of-two scale mode (the scales Blackwell's UE8M0 microscaling
  formats hold; the pages point to Blackwell microscaling as the direction
  of FP8 hardware): s = the smallest power of two with amax / s <= 448, by a
  plain search in ``fp8bs_oracle.c``; codes and GEMM as above.
* Normalization fused with the 1x128 cast (RMSNorm or LayerNorm, bf16
  output, then the activation quantizer): "How I Improved My Deepseek In In
  The Future", paragraph of hardware suggestions (fusion of layer
  normalization and FP8 cast). Row statistics in float64 rounded once to
  binary32; the elementwise part as binary32 numpy operations. Since a float
  sum has no single evaluation order, the oracle also enumerates, from its
  own statistics outward, every binary32 statistic inside a given error
  interval and the codes each gives (``norm_stat_rings``, ``norm_rows_at``);
  it never takes statistics from the code under test.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bs_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_fp8bs.so")

# Flags that keep every float operation a single IEEE binary32 operation.
_CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-fexcess-precision=standard", "-fno-math-errno"]


def build(force: bool = False) -> str:
    """Compile the C half of the oracle with gcc (no CUDA involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp"
        subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        i64 = ctypes.c_int64
        L.fp8o_e4m3_decode.restype = ctypes.c_double
        L.fp8o_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.fp8o_e4m3_encode.restype = ctypes.c_uint8
        L.fp8o_e4m3_encode.argtypes = [ctypes.c_float]
        L.fp8o_group_scale.restype = ctypes.c_float
        L.fp8o_group_scale.argtypes = [ctypes.c_float]
        L.fp8o_quantize_value.restype = ctypes.c_uint8
        L.fp8o_quantize_value.argtypes = [ctypes.c_float, ctypes.c_float]
        L.fp8o_quantize_act_1x128.restype = None
        L.fp8o_quantize_act_1x128.argtypes = [u16p, i64, i64, i64, u8p, i64, f32p]
        L.fp8o_quantize_weight_128x128.restype = None
        L.fp8o_quantize_weight_128x128.argtypes = [u16p, i64, i64, i64, u8p, i64, f32p]
        L.fp8o_quantize_pairs.restype = None
        L.fp8o_quantize_pairs.argtypes = [u16p, u16p, i64, u8p, f32p]
        L.fp8o_group_scale_pow2.restype = ctypes.c_float
        L.fp8o_group_scale_pow2.argtypes = [ctypes.c_float]
        L.fp8o_quantize_act_1x128_pow2.restype = None
        L.fp8o_quantize_act_1x128_pow2.argtypes = [u16p, i64, i64, i64, u8p, i64, f32p]
        L.fp8o_quantize_weight_128x128_pow2.restype = None
        L.fp8o_quantize_weight_128x128_pow2.argtypes = [u16p, i64, i64, i64, u8p, i64, f32p]
        L.fp8o_quantize_pairs_mode.restype = None
        L.fp8o_quantize_pairs_mode.argtypes = [u16p, u16p, i64, u8p, f32p, ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"] or a.ndim == 0
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ---------------------------------------------------------------------------
# E4M3 codec
# ---------------------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return lib().fp8o_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(y: float) -> int:
    return int(lib().fp8o_e4m3_encode(float(np.float32(y))))


def e4m3_table() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for 0x7F and 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def group_scale(amax: float) -> np.float32:
    return np.float32(lib().fp8o_group_scale(float(np.float32(amax))))


def quantize_value(x: float, s: float) -> int:
    return int(lib().fp8o_quantize_value(float(np.float32(x)), float(np.float32(s))))


# ---------------------------------------------------------------------------
# Quantizers. Inputs are bf16 bit patterns held as uint16 arrays.
# ---------------------------------------------------------------------------

def quantize_act_1x128(x_bits: np.ndarray, pow2: bool = False):
    """x_bits: uint16 [M, K] (bf16 patterns) -> (q uint8 [M, K], s float32 [M, K/128]).
    pow2: power-of-two scales (group_scale_pow2) instead of amax / 448."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    assert K % 128 == 0
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, K // 128), dtype=np.float32)
    if M and K:
        fn = lib().fp8o_quantize_act_1x128_pow2 if pow2 else lib().fp8o_quantize_act_1x128
        fn(_ptr(x_bits, ctypes.c_uint16), M, K, K, _ptr(q, ctypes.c_uint8), K, _ptr(s, ctypes.c_float))
    return q, s


def quantize_weight_128x128(w_bits: np.ndarray, pow2: bool = False):
    """w_bits: uint16 [N, K] -> (q uint8 [N, K], s float32 [ceil(N/128), K/128])."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = w_bits.shape
    assert K % 128 == 0
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty(((N + 127) // 128, K // 128), dtype=np.float32)
    if N and K:
        fn = lib().fp8o_quantize_weight_128x128_pow2 if pow2 else lib().fp8o_quantize_weight_128x128
        fn(_ptr(w_bits, ctypes.c_uint16), N, K, K, _ptr(q, ctypes.c_uint8), K, _ptr(s, ctypes.c_float))
    return q, s


def group_scale_pow2(amax: float) -> np.float32:
    return np.float32(lib().fp8o_group_scale_pow2(float(np.float32(amax))))


def quantize_pairs(amax_bits: np.ndarray, x_bits: np.ndarray, pow2: bool = False):
    """Codes of x under the scale of amax, element by element."""
    amax_bits = np.ascontiguousarray(amax_bits, dtype=np.uint16).ravel()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16).ravel()
    n = x_bits.size
    q = np.empty(n, dtype=np.uint8)
    s = np.empty(n, dtype=np.float32)
    if n:
        lib().fp8o_quantize_pairs_mode(_ptr(amax_bits, ctypes.c_uint16), _ptr(x_bits, ctypes.c_uint16),
                                       n, _ptr(q, ctypes.c_uint8), _ptr(s, ctypes.c_float), int(pow2))
    return q, s


# ---------------------------------------------------------------------------
# Dequantization and the GEMM (float64).
# ---------------------------------------------------------------------------

_TABLE = None


def _table() -> np.ndarray:
    global _TABLE
    if _TABLE is None:
        _TABLE = e4m3_table()
    return _TABLE


def dequant_act(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """A_hat[m, k] = value(q[m, k]) * s[m, k // 128], exact in float64."""
    M, K = q.shape
    return _table()[q] * np.repeat(s.astype(np.float64), 128, axis=1)[:, :K]


def dequant_weight(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """W_hat[n, k] = value(q[n, k]) * s[n // 128, k // 128], exact in float64."""
    N, K = q.shape
    sf = np.repeat(np.repeat(s.astype(np.float64), 128, axis=0), 128, axis=1)[:N, :K]
    return _table()[q] * sf


def gemm(qa, sa, qw, sw):
    """C_or = A_hat @ W_hat^T and B = |A_hat| @ |W_hat|^T, both float64 [M, N]."""
    A = dequant_act(qa, sa)
    W = dequant_weight(qw, sw)
    return A @ W.T, np.abs(A) @ np.abs(W).T


def gemm_entries(qa, sa, qw, sw, rows, cols):
    """C_or and B at the listed (row, col) pairs only, one dot product each."""
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    A = dequant_act(qa[rows], sa[rows])
    W = dequant_weight_rows(qw, sw, cols)
    prod = A * W
    return prod.sum(axis=1), np.abs(prod).sum(axis=1)


def dequant_weight_rows(qw, sw, rows):
    """W_hat for the listed output channels."""
    rows = np.asarray(rows)
    K = qw.shape[1]
    sf = np.repeat(sw.astype(np.float64)[rows // 128], 128, axis=1)[:, :K]
    return _table()[qw[rows]] * sf


def grouped_gemm(qa, sa, offsets, qw, sw):
    """Per expert e: rows offsets[e]:offsets[e+1] of A times W_e^T.

    qw: uint8 [E, N, K]; sw: float32 [E, ceil(N/128), K/128]."""
    E = len(offsets) - 1
    total = int(offsets[-1])
    N = qw.shape[1]
    C = np.zeros((total, N), dtype=np.float64)
    B = np.zeros((total, N), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            C[lo:hi], B[lo:hi] = gemm(qa[lo:hi], sa[lo:hi], qw[e], sw[e])
    return C, B


def tolerance(C_or: np.ndarray, B: np.ndarray, out_bf16: bool) -> np.ndarray:
    """Elementwise acceptance bound for a GPU result against C_or."""
    tol = 2e-5 * B + 1e-6
    if out_bf16:
        tol = tol + np.abs(C_or) * 2.0 ** -8
    return tol


# ---------------------------------------------------------------------------
# Normalization fused with the 1x128 cast.
#
# "How I Improved My Deepseek In In The Future", paragraph of hardware
# suggestions: a warp-level cast instruction would allow the layer
# normalization and the FP8 cast to be fused. Reading taken here: the fused
# producer computes exactly what a normalization layer with a bf16 output
# followed by the 1x128 activation quantizer computes. Two kinds:
#   RMSNorm   y = x * rstd * gamma (+ beta),   rstd = 1/sqrt(mean(x^2) + eps)
#   LayerNorm y = (x - mu) * rstd * gamma (+ beta),
#             mu = mean(x), rstd = 1/sqrt(mean((x - mu)^2) + eps)
# Row statistics are exact in float64 and then rounded once to binary32 (the
# precision the layer stores them in). The elementwise part is written as
# binary32 operations in the order above (subtract, multiply by rstd,
# multiply by gamma, add beta), each rounded to nearest, and the result is
# rounded to bf16 (nearest-even) before the 1x128 quantizer sees it.
# ---------------------------------------------------------------------------
NORM_RMS = 0
NORM_LAYER = 1


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the same values as float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(y: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, rounded to nearest, ties to even.

    The 16 low bits are dropped after adding half an ulp of the result,
    less one when the kept part is even (so that an exact half goes to the
    even neighbour). Finite inputs only."""
    u = np.ascontiguousarray(y, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep_odd = (u >> 16) & 1
    return ((u + 0x7FFF + keep_odd) >> 16).astype(np.uint16)


def norm_stats(x_bits: np.ndarray, kind: int, eps: float):
    """Row statistics (mu, rstd) as float32 [M]; mu is 0 for RMSNorm."""
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    eps64 = float(np.float32(eps))
    M, K = x.shape
    if kind == NORM_RMS:
        mu = np.zeros(M)
        var = (x * x).sum(axis=1) / K
    elif kind == NORM_LAYER:
        mu = x.sum(axis=1) / K
        d = x - mu[:, None]
        var = (d * d).sum(axis=1) / K
    else:
        raise ValueError(f"unknown normalization kind {kind}")
    rstd = 1.0 / np.sqrt(var + eps64)
    return mu.astype(np.float32), rstd.astype(np.float32)


def norm_apply(x_bits, gamma_bits, beta_bits, kind: int, mu32, rstd32) -> np.ndarray:
    """bf16 patterns of the normalized rows, given binary32 row statistics."""
    x = bf16_bits_to_f32(x_bits)
    mu32 = np.asarray(mu32, dtype=np.float32)[:, None]
    rstd32 = np.asarray(rstd32, dtype=np.float32)[:, None]
    d = x - mu32 if kind == NORM_LAYER else x
    t = d * rstd32
    u = t * bf16_bits_to_f32(gamma_bits)[None, :]
    y = u + bf16_bits_to_f32(beta_bits)[None, :] if beta_bits is not None else u
    return f32_to_bf16_bits(y)


def norm_quantize_act_1x128(x_bits, gamma_bits, beta_bits, kind: int, eps: float):
    """Normalize each row with the oracle's own statistics, round to bf16,
    quantize in 1x128 tiles.

    Returns (q uint8 [M, K], s float32 [M, K/128], mu float32 [M],
    rstd float32 [M], y uint16 [M, K])."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    mu32, rstd32 = norm_stats(x_bits, kind, eps)
    y = norm_apply(x_bits, gamma_bits, beta_bits, kind, mu32, rstd32)
    q, s = quantize_act_1x128(y)
    return q, s, mu32, rstd32, y


# ---------------------------------------------------------------------------
# Admissible row statistics.
#
# A float sum has no single correct evaluation order, so a normalization
# layer computed in binary32 may return statistics a few units in the last
# place away from the correctly rounded ones above; every such binary32 value
# inside a proven error interval is an acceptable statistic, and the codes it
# leads to are acceptable codes. These helpers enumerate those values from the
# oracle's own statistics outward (nearest first) and evaluate the row under
# each of them with the same elementwise steps as above.
# ---------------------------------------------------------------------------

def f32_step(v32, steps):
    """The binary32 value `steps` representable numbers above v32 (below for
    negative steps), walking through zero; finite values only."""
    v = np.asarray(v32, dtype=np.float32)
    bits = v.view(np.int32).astype(np.int64)
    key = np.where(bits >= 0, bits, -(bits & 0x7FFFFFFF))        # monotone in the value
    key = key + np.asarray(steps, dtype=np.int64)
    out = np.where(key >= 0, key, (-key) | 0x80000000).astype(np.uint32)
    return out.view(np.float32)


def norm_stat_rings(mu32: float, rstd32: float, kind: int, mu_abs: float, rstd_rel: float,
                    max_ring: int):
    """Candidate binary32 statistics around (mu32, rstd32), ring by ring.

    Ring d holds the pairs (mu32 stepped by i, rstd32 stepped by j) with
    max(|i|, |j|) = d that lie within |mu - mu32| <= mu_abs and
    |rstd - rstd32| <= rstd_rel * rstd32 (mu stays 0 for RMSNorm). Yields
    (d, mu array, rstd array) for d = 0, 1, ... while a ring has members and
    d <= max_ring."""
    mu32 = np.float32(mu32)
    rstd32 = np.float32(rstd32)
    r_lim = float(rstd_rel) * float(rstd32)
    for d in range(max_ring + 1):
        if d == 0:
            ii = np.zeros(1, np.int64)
            jj = np.zeros(1, np.int64)
        elif kind == NORM_RMS:
            ii = np.zeros(2, np.int64)
            jj = np.array([-d, d], np.int64)
        else:
            r = np.arange(-d, d + 1, dtype=np.int64)
            ii = np.concatenate([np.full(r.size, -d), np.full(r.size, d), r[1:-1], r[1:-1]])
            jj = np.concatenate([r, r, np.full(r.size - 2, -d), np.full(r.size - 2, d)])
        mu_c = f32_step(np.full(ii.size, mu32), ii) if kind == NORM_LAYER else np.zeros(ii.size, np.float32)
        r_c = f32_step(np.full(jj.size, rstd32), jj)
        ok = np.abs(r_c.astype(np.float64) - float(rstd32)) <= r_lim
        if kind == NORM_LAYER:
            ok &= np.abs(mu_c.astype(np.float64) - float(mu32)) <= float(mu_abs)
        if not ok.any():
            return
        yield d, mu_c[ok], r_c[ok]


def norm_rows_at(x_row_bits, gamma_bits, beta_bits, kind: int, mu32, rstd32):
    """One row normalized and quantized under each candidate (mu32[i],
    rstd32[i]): q uint8 [n, K], s float32 [n, K/128]."""
    x_row_bits = np.ascontiguousarray(x_row_bits, dtype=np.uint16).ravel()
    n = len(rstd32)
    xs = np.broadcast_to(x_row_bits, (n, x_row_bits.size))
    y = norm_apply(xs, gamma_bits, beta_bits, kind, mu32, rstd32)
    return quantize_act_1x128(y)
