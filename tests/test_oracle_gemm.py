"""Pins for the oracle's dequantize-then-contract GEMM and its grouped form.

Each case fixes the answer by something other than the oracle: a closed form,
a special structure (identity, one-hot with a permutation), or exact rational
arithmetic on a small brute-force case. A transposed operand, a wrong scale
index or a dropped K chunk fails at least one of them."""
from fractions import Fraction

import numpy as np
import pytest

from fp8_fine_grained_17_b300 import workloads as wl


def _q(orc, a, w):
    qa, sa = orc.quantize_act_1x128(wl.bf16_bits(a))
    qw, sw = orc.quantize_weight_128x128(wl.bf16_bits(w))
    return qa, sa, qw, sw


def test_identity_weight(orc):
    rng = np.random.default_rng(10)
    M, K = 64, 512
    a = rng.standard_normal((M, K)).astype(np.float32)
    w = np.eye(K, dtype=np.float32)
    qa, sa, qw, sw = _q(orc, a, w)
    # diagonal blocks: amax 1 -> s = fl32(1/448), code 0x7E; off-diagonal: zero blocks
    s1 = np.float32(1.0) / np.float32(448.0)
    for nb in range(4):
        for kb in range(4):
            assert sw[nb, kb] == (s1 if nb == kb else np.float32(1.0))
    assert np.all(np.diag(qw) == 0x7E)
    C, B = orc.gemm(qa, sa, qw, sw)
    A_hat = orc.dequant_act(qa, sa)
    expect = A_hat * (448.0 * float(s1))
    assert np.allclose(C, expect, rtol=1e-15, atol=0)
    assert np.allclose(B, np.abs(expect), rtol=1e-15, atol=0)


def test_one_hot_permutation(orc):
    rng = np.random.default_rng(11)
    M, N, K = 32, 384, 256
    perm = rng.integers(0, K, N)
    vals = rng.uniform(0.5, 4.0, N).astype(np.float32)
    a = rng.standard_normal((M, K)).astype(np.float32)
    w = np.zeros((N, K), dtype=np.float32)
    w[np.arange(N), perm] = vals
    qa, sa, qw, sw = _q(orc, a, w)
    C, _ = orc.gemm(qa, sa, qw, sw)
    A_hat = orc.dequant_act(qa, sa)
    table = orc.e4m3_table()
    for n in range(N):
        w_hat = table[qw[n, perm[n]]] * float(sw[n // 128, perm[n] // 128])
        assert np.allclose(C[:, n], A_hat[:, perm[n]] * w_hat, rtol=1e-15, atol=0)


def test_closed_form_constant_rows(orc):
    M, N, K = 8, 256, 512
    a = np.ones((M, K), dtype=np.float32)
    w = ((np.arange(N) % 3) + 1).astype(np.float32)[:, None].repeat(K, axis=1)
    qa, sa, qw, sw = _q(orc, a, w)
    s_a = np.float32(1.0) / np.float32(448.0)
    s_w = np.float32(3.0) / np.float32(448.0)
    assert np.all(sa == s_a) and np.all(sw == s_w)
    # 1/s_w = 149.33 -> 144, 2/s_w = 298.67 -> 288, 3/s_w -> 448 (E4M3 grid)
    w_hat = np.array([144.0, 288.0, 448.0]) * float(s_w)
    C, _ = orc.gemm(qa, sa, qw, sw)
    expect = K * (448.0 * float(s_a)) * w_hat[np.arange(N) % 3]
    assert np.allclose(C, np.broadcast_to(expect, (M, N)), rtol=1e-13, atol=0)


def test_per_chunk_scales(orc):
    """A chunk kb holds the constant 2^kb, so each chunk has its own scale;
    using one chunk's scale for all of them changes the sum."""
    M, N, K = 4, 128, 512
    a = np.concatenate([np.full((M, 128), 2.0 ** kb, np.float32) for kb in range(4)], axis=1)
    w = np.ones((N, K), dtype=np.float32)
    qa, sa, qw, sw = _q(orc, a, w)
    s1 = float(np.float32(1.0) / np.float32(448.0))
    expect = 128 * (448.0 * s1) ** 2 * (1 + 2 + 4 + 8)
    C, _ = orc.gemm(qa, sa, qw, sw)
    assert np.allclose(C, expect, rtol=1e-14, atol=0)


def test_only_one_chunk_nonzero(orc):
    rng = np.random.default_rng(12)
    M, N, K = 4, 128, 512
    a = np.zeros((M, K), np.float32)
    a[:, 128:256] = rng.standard_normal((M, 128))
    w = rng.standard_normal((N, K)).astype(np.float32)
    qa, sa, qw, sw = _q(orc, a, w)
    C, _ = orc.gemm(qa, sa, qw, sw)
    A_hat = orc.dequant_act(qa, sa)[:, 128:256]
    W_hat = orc.dequant_weight(qw, sw)[:, 128:256]
    assert np.allclose(C, A_hat @ W_hat.T, rtol=1e-14, atol=1e-300)


def test_brute_force_exact_rational(orc):
    """4x128x128 with exact rational sums; float64 error within gamma_K * B."""
    rng = np.random.default_rng(13)
    M, N, K = 4, 128, 128
    a = (rng.standard_normal((M, K)) * 3).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    qa, sa, qw, sw = _q(orc, a, w)
    C, B = orc.gemm(qa, sa, qw, sw)
    table = orc.e4m3_table()
    gamma = K * 2.0 ** -53 / (1 - K * 2.0 ** -53)
    for m in range(M):
        for n in range(0, N, 5):
            exact = sum(Fraction(table[qa[m, k]]) * Fraction(float(sa[m, 0])) *
                        Fraction(table[qw[n, k]]) * Fraction(float(sw[0, 0]))
                        for k in range(K))
            babs = sum(abs(Fraction(table[qa[m, k]]) * Fraction(table[qw[n, k]])) for k in range(K)) \
                * Fraction(float(sa[m, 0])) * Fraction(float(sw[0, 0]))
            assert abs(Fraction(C[m, n]) - exact) <= Fraction(gamma) * babs
            assert abs(Fraction(B[m, n]) - babs) <= Fraction(gamma) * babs


def test_gemm_entries_match_full(orc):
    rng = np.random.default_rng(14)
    a = rng.standard_normal((40, 256)).astype(np.float32)
    w = rng.standard_normal((256, 256)).astype(np.float32)
    qa, sa, qw, sw = _q(orc, a, w)
    C, B = orc.gemm(qa, sa, qw, sw)
    rows = rng.integers(0, 40, 50)
    cols = rng.integers(0, 256, 50)
    c, b = orc.gemm_entries(qa, sa, qw, sw, rows, cols)
    assert np.allclose(c, C[rows, cols], rtol=1e-12, atol=1e-300)
    assert np.allclose(b, B[rows, cols], rtol=1e-12, atol=1e-300)


def test_grouped_one_hot_experts(orc):
    """Expert e has W_e = (e+1) * one-hot(n -> (n + e) mod K); empty experts allowed."""
    rng = np.random.default_rng(15)
    counts = [3, 0, 5, 1]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    N, K = 128, 256
    a = rng.standard_normal((int(off[-1]), K)).astype(np.float32)
    qa, sa = orc.quantize_act_1x128(wl.bf16_bits(a))
    qws, sws = [], []
    for e in range(len(counts)):
        w = np.zeros((N, K), np.float32)
        w[np.arange(N), (np.arange(N) + e) % K] = e + 1
        q, s = orc.quantize_weight_128x128(wl.bf16_bits(w))
        qws.append(q)
        sws.append(s)
    qw, sw = np.stack(qws), np.stack(sws)
    C, _ = orc.grouped_gemm(qa, sa, off, qw, sw)
    A_hat = orc.dequant_act(qa, sa)
    for e in range(len(counts)):
        s = float(np.float32(e + 1) / np.float32(448.0))
        for r in range(off[e], off[e + 1]):
            expect = A_hat[r, (np.arange(N) + e) % K] * 448.0 * s
            assert np.allclose(C[r], expect, rtol=1e-15, atol=0)


def test_tolerance_formula(orc):
    C = np.array([1.0, -2.0])
    B = np.array([3.0, 4.0])
    t32 = orc.tolerance(C, B, out_bf16=False)
    t16 = orc.tolerance(C, B, out_bf16=True)
    assert np.allclose(t32, [2e-5 * 3 + 1e-6, 2e-5 * 4 + 1e-6], rtol=0, atol=0)
    assert np.allclose(t16, t32 + np.array([1.0, 2.0]) / 256, rtol=0, atol=0)
