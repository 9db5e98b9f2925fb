"""GPU parity of the two quantizers against the oracle: codes and scales must
be bit-identical. Covers ragged and degenerate shapes, the full
activation-quantize workload [16384, 7168] with 0.5% outlier channels, and
every (bf16 amax, bf16 x) pair with |x| <= amax."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import fp8bs
from fp8_fine_grained_17_b300 import workloads as wl
from helpers import check_codes, gpu_quant_act, gpu_quant_weight, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(1, 128), (3, 384), (17, 1024), (129, 640), (1000, 7168)])
def test_act_quant_shapes(orc, M, K):
    rng = np.random.default_rng(M * 7 + K)
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(10.0) ** rng.integers(-6, 6, (M, 1))
    x[0, :128] = 0.0                     # an all-zero group -> s = 1
    if M > 2:
        x[2, 5] = -0.0
        x[1, 1] = 1e30                   # bf16-range outlier
    bits = wl.bf16_bits(x)
    q, s = gpu_quant_act(bits)
    check_codes(q, s, *orc.quantize_act_1x128(bits))


def test_act_quant_strided(orc):
    """Row strides larger than K on input and output."""
    rng = np.random.default_rng(21)
    M, K, ldx, ldq = 37, 256, 384, 272
    bits = wl.bf16_bits(rng.standard_normal((M, ldx)).astype(np.float32))
    x = to_dev_bf16(bits)[:, :K]
    qbuf = torch.full((M, ldq), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    fp8bs.fp8bs_quantize_act_1x128(x, qbuf[:, :K], s)
    q_or, s_or = orc.quantize_act_1x128(np.ascontiguousarray(bits[:, :K]))
    check_codes(qbuf[:, :K].contiguous(), s, q_or, s_or)
    assert torch.all(qbuf[:, K:] == 0xAB)          # nothing written past K


def test_act_quant_empty():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = fp8bs.quantize_act(x)
    assert q.shape == (0, 256) and s.shape == (0, 2)


def test_act_quant_full_workload(orc):
    """[16384, 7168] bf16 ~ N(0,1) with 36 channels x100: every code and scale."""
    d = wl.cfg1(0)
    q, s = gpu_quant_act(d.a_bits)
    check_codes(q, s, *orc.quantize_act_1x128(d.a_bits))


@pytest.mark.parametrize("N,K", [(128, 128), (300, 256), (1, 512), (7168, 2048)])
def test_weight_quant_shapes(orc, N, K):
    rng = np.random.default_rng(N + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[N // 2, K // 3] = 3.0
    if N >= 256:
        w[128:256, 128:256] = 0.0        # an all-zero block
    bits = wl.bf16_bits(w)
    q, s = gpu_quant_weight(bits)
    check_codes(q, s, *orc.quantize_weight_128x128(bits))


def _pair_rows(a_lo: int, a_hi: int) -> np.ndarray:
    """Rows [amax, x_1..x_127] covering every bf16 x with |x| <= amax for each
    positive finite bf16 amax pattern in [a_lo, a_hi); short rows padded with 0."""
    A = np.arange(a_lo, a_hi, dtype=np.int64)
    n_x = 2 * (A + 1)                                # +0..amax and -0..-amax
    n_rows = (n_x + 126) // 127
    row_a = np.repeat(A, n_rows)
    start = np.concatenate([[0], np.cumsum(n_rows)[:-1]])
    local = np.arange(row_a.size, dtype=np.int64) - np.repeat(start, n_rows)
    j = local[:, None] * 127 + np.arange(127, dtype=np.int64)[None, :]
    a = row_a[:, None]
    x = np.where(j <= a, j, 0x8000 + j - a - 1)
    x = np.where(j < 2 * (a + 1), x, 0)
    rows = np.empty((row_a.size, 128), dtype=np.uint16)
    rows[:, 0] = row_a
    rows[:, 1:] = x
    return rows


# The activation quantizer streams large contiguous inputs through a shared-
# memory ring of bulk copies and takes smaller ones through registers; both
# paths are checked on every pair.
RING_MIN_GROUPS = 1 << 19


@pytest.mark.slow
def test_exhaustive_amax_x_pairs(orc):
    """All ~1.07e9 (amax, x) pairs: the code of one element depends only on its
    group's amax and its own value, so this covers the quantizer's whole
    input space, including subnormal scales and the small-amax path. Each
    slice runs through both kernel paths: alone (register path) and padded
    with all-zero groups to the ring path's minimum size."""
    edges = np.linspace(1, 0x7F80, 49).astype(np.int64)
    pool = ThreadPoolExecutor(max_workers=8)
    total = 0
    for lo, hi in zip(edges[:-1], edges[1:]):
        rows = _pair_rows(int(lo), int(hi))
        total += rows.size
        assert rows.shape[0] < RING_MIN_GROUPS
        q, s = gpu_quant_act(rows)
        padded = np.zeros((RING_MIN_GROUPS, 128), dtype=np.uint16)
        padded[:rows.shape[0]] = rows
        qp, sp = gpu_quant_act(padded)
        parts = np.array_split(np.arange(rows.shape[0]), 8)
        res = list(pool.map(lambda ix: orc.quantize_act_1x128(rows[ix]), parts))
        q_or = np.concatenate([r[0] for r in res])
        s_or = np.concatenate([r[1] for r in res])
        check_codes(q, s, q_or, s_or)
        check_codes(qp[:rows.shape[0]], sp[:rows.shape[0]], q_or, s_or)
        assert torch.all(qp[rows.shape[0]:] == 0) and torch.all(sp[rows.shape[0]:] == 1.0)
    pool.shutdown()
    assert total > 1.07e9


# Large contiguous pairs run the ring kernel (activation chunks by bulk copy,
# weight blocks by 2-D TMA): the bench shape, a ragged last activation chunk
# with a partial last weight block (N = 3999), and weights alone (N = 8191);
# the small and strided ones run the one-unit-per-CTA pair kernel.
@pytest.mark.parametrize("M,K,N,Kw,strided", [
    (4096, 7168, 4096, 7168, False), (2050, 7168, 3999, 7168, False), (0, 128, 8191, 4096, False),
    (1, 128, 300, 256, False), (37, 384, 0, 128, False),
    (0, 128, 129, 512, False), (257, 1152, 640, 896, True),
])
def test_pair_quantizer_matches_separate(orc, M, K, N, Kw, strided):
    """One launch of both quantizers: codes and scales bit-identical to the
    oracle (and so to the separate kernels)."""
    rng = np.random.default_rng(M + K + N + Kw)
    a_bits, _ = wl.activations(rng, M, K, 100.0)
    w_bits = wl.weights(rng, N, Kw)
    pad = 64 if strided else 0
    xs = torch.zeros((M, K + pad), dtype=torch.bfloat16, device="cuda")
    xs[:, :K] = wl.bits_to_torch(a_bits).cuda()
    ws = torch.zeros((N, Kw + pad), dtype=torch.bfloat16, device="cuda")
    ws[:, :Kw] = wl.bits_to_torch(w_bits).cuda()
    qxs = torch.zeros((M, K + pad), dtype=torch.uint8, device="cuda")
    qws = torch.zeros((N, Kw + pad), dtype=torch.uint8, device="cuda")
    sx = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    sw = torch.empty(((N + 127) // 128, Kw // 128), dtype=torch.float32, device="cuda")
    fp8bs.fp8bs_quantize_act_and_weight(xs[:, :K], qxs[:, :K], sx, ws[:, :Kw], qws[:, :Kw], sw)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    if M:
        q_o, s_o = orc.quantize_act_1x128(a_bits)
        check_codes(qxs[:, :K], sx, q_o, s_o)
    if N:
        q_o, s_o = orc.quantize_weight_128x128(w_bits)
        check_codes(qws[:, :Kw], sw, q_o, s_o)
    if pad:
        assert torch.all(qxs[:, K:] == 0).item() and torch.all(qws[:, Kw:] == 0).item()




def _random_pair_cases(n=12, seed=99):
    """Seeded activation and weight shapes for the one-launch pair: empty
    sides, partial weight blocks, padded strides, and sizes on both sides of
    the ring kernel's threshold."""
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        M = int(rng.choice([0, 1, 77, 513, 2048, 3000]))
        K = 128 * int(rng.choice([1, 5, 16, 56, 64]))
        N = int(rng.choice([0, 1, 129, 1000, 4096, 4999]))
        Kw = 128 * int(rng.choice([1, 7, 16, 56]))
        strided = bool(rng.random() < 0.3)
        cases.append((M, K, N, Kw, strided))
    return cases


@pytest.mark.parametrize("M,K,N,Kw,strided", _random_pair_cases())
def test_pair_quantizer_random(orc, M, K, N, Kw, strided):
    test_pair_quantizer_matches_separate(orc, M, K, N, Kw, strided)

# ---------------------------------------------------------------- power-of-two scales

def _pow2_rows():
    """One row per positive finite bf16 amax: [amax, -amax, -0, +0, then 124
    seeded values with |x| <= amax spread over the binades below it]."""
    rng = np.random.default_rng(31)
    amax = np.arange(1, 0x7F80, dtype=np.uint16)
    rows = np.zeros((amax.size, 128), dtype=np.uint16)
    rows[:, 0] = amax
    rows[:, 1] = amax | 0x8000
    rows[:, 2] = 0x8000
    frac = rng.random((amax.size, 124)) * np.exp2(-rng.integers(0, 40, (amax.size, 124)))
    vals = wl.bits_to_f32(amax)[:, None] * frac.astype(np.float32)
    vals *= np.where(rng.random(vals.shape) < 0.5, -1.0, 1.0).astype(np.float32)
    b = wl.bf16_bits(vals)
    mag = b & 0x7FFF
    b = np.where(mag > amax[:, None], (b & 0x8000) | amax[:, None], b)   # rounding may pass amax
    rows[:, 4:] = b
    return rows


def test_pow2_act_every_amax_both_paths(orc):
    rows = _pow2_rows()
    q_or, s_or = orc.quantize_act_1x128(rows, pow2=True)
    x = to_dev_bf16(rows)
    q, s = fp8bs.quantize_act(x, pow2=True)
    check_codes(q, s, q_or, s_or)
    padded = np.zeros((RING_MIN_GROUPS, 128), dtype=np.uint16)
    padded[:rows.shape[0]] = rows
    qp, sp = fp8bs.quantize_act(to_dev_bf16(padded), pow2=True)
    check_codes(qp[:rows.shape[0]], sp[:rows.shape[0]], q_or, s_or)


@pytest.mark.parametrize("N,K", [(128, 128), (300, 256), (7168, 2048)])
def test_pow2_weight_shapes(orc, N, K):
    rng = np.random.default_rng(N + K + 1)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[N // 2, K // 3] = 3.0
    bits = wl.bf16_bits(w)
    q, s = fp8bs.quantize_weight(to_dev_bf16(bits), pow2=True)
    check_codes(q, s, *orc.quantize_weight_128x128(bits, pow2=True))


def test_pow2_act_full_workload(orc):
    d = wl.cfg1(0)
    q, s = fp8bs.quantize_act(to_dev_bf16(d.a_bits), pow2=True)
    check_codes(q, s, *orc.quantize_act_1x128(d.a_bits, pow2=True))
