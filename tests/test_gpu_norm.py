"""RMSNorm / LayerNorm fused with the 1x128 cast on the GPU against the oracle.

The row statistics come from parallel binary32 sums, so they are checked
against the oracle's correctly rounded statistics within the proven bound of
that summation. The codes and scales of each row must then equal the oracle's
row at some binary32 statistic inside that bound; the oracle enumerates those
statistics from its own values outward, so nothing computed by the kernel
enters the oracle. How many rows needed a non-central statistic is printed."""
import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import fp8bs
from fp8_fine_grained_17_b300 import workloads as wl
from oracle import oracle as orc

from helpers import check_norm_rows, to_dev_bf16

pytestmark = pytest.mark.gpu


def run_norm(x_bits, g_bits, b_bits, kind, eps, ldx=None, ldq=None):
    M, K = x_bits.shape
    ldx = ldx or K
    ldq = ldq or K
    xs = torch.zeros((M, ldx), dtype=torch.bfloat16, device="cuda")
    xs[:, :K] = to_dev_bf16(x_bits)
    x = xs[:, :K]
    g = to_dev_bf16(g_bits)
    b = to_dev_bf16(b_bits) if b_bits is not None else None
    qs = torch.full((M, ldq), 0xA5, dtype=torch.uint8, device="cuda")
    q = qs[:, :K]
    s = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    mean = torch.full((M,), -7.0, dtype=torch.float32, device="cuda")
    rstd = torch.empty(M, dtype=torch.float32, device="cuda")
    fp8bs.fp8bs_norm_quantize_act_1x128(x, g, b, kind, eps, q, s, mean, rstd)
    assert fp8bs.fp8bs_last_device_error() == fp8bs.OK
    if ldq > K:   # padding bytes untouched
        assert torch.all(qs[:, K:] == 0xA5).item()
    return q, s, mean.cpu().numpy(), rstd.cpu().numpy()


def check_norm(x_bits, g_bits, b_bits, kind, eps, q, s, mean_k, rstd_k, rows=None):
    """Compare the listed rows (all by default); print the non-central count."""
    q = q.cpu().numpy() if torch.is_tensor(q) else q
    s = s.cpu().numpy() if torch.is_tensor(s) else s
    if rows is not None:
        x_bits = x_bits[rows]
        q, s = q[rows], s[rows]
        mean_k, rstd_k = mean_k[rows], rstd_k[rows]
    n, off, ring = check_norm_rows(orc, x_bits, g_bits, b_bits, kind, eps, q, s, mean_k, rstd_k)
    print(f"norm kind={kind} K={x_bits.shape[1]}: {n} rows, {off} matched a non-central "
          f"statistic (farthest {ring} ulp)")
    return off


SHAPES = [(1, 128), (5, 384), (37, 1024), (64, 2048), (33, 4096), (19, 5120), (70, 7168),
          (9, 8192), (6, 12288), (3, 16384), (2, 24576), (2, 40960), (1, 65536)]


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
@pytest.mark.parametrize("M,K", SHAPES)
def test_norm_quant_shapes(kind, M, K):
    n = wl.norm(M, K, seed=M * 7 + K + kind, with_beta=(K // 128) % 2 == 1)
    q, s, mean, rstd = run_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6)
    check_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6, q, s, mean, rstd)


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
def test_norm_quant_strided(kind):
    n = wl.norm(45, 1152, seed=3, with_beta=True)
    q, s, mean, rstd = run_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-5, ldx=1160, ldq=1168)
    check_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-5, q, s, mean, rstd)


def test_norm_quant_degenerate_rows():
    # All-zero rows (RMSNorm, eps > 0: y = 0, every code 0, scale 1) and
    # constant rows (LayerNorm: y = beta), mixed with ordinary rows.
    n = wl.norm(12, 768, seed=5, with_beta=True)
    x = n.x_bits.copy()
    x[[0, 4, 11]] = 0
    x[[2, 7]] = wl.bf16_bits(np.full(768, -3.25, np.float32))
    for kind in (orc.NORM_RMS, orc.NORM_LAYER):
        q, s, mean, rstd = run_norm(x, n.gamma_bits, n.beta_bits, kind, 1e-6)
        check_norm(x, n.gamma_bits, n.beta_bits, kind, 1e-6, q, s, mean, rstd)
    q, s, _, _ = run_norm(x, n.gamma_bits, None, orc.NORM_RMS, 1e-6)
    assert torch.all(q[[0, 4, 11]] == 0).item() and torch.all(s[[0, 4, 11]] == 1.0).item()


def test_norm_quant_matches_unfused_gpu_quantizer():
    # Where the fused kernel's rows equal the oracle's central rows (checked
    # first), the 1x128 quantizer kernel applied to the oracle's normalized
    # bf16 rows gives the same codes and scales: the fusion changes nothing
    # but the memory traffic.
    n = wl.norm(96, 7168, seed=8, with_beta=False)
    q, s, mean, rstd = run_norm(n.x_bits, n.gamma_bits, None, orc.NORM_RMS, 1e-6)
    q_c, s_c, _, _, y = orc.norm_quantize_act_1x128(n.x_bits, n.gamma_bits, None, orc.NORM_RMS, 1e-6)
    rows = np.flatnonzero(np.all(q.cpu().numpy() == q_c, axis=1) &
                          np.all(s.cpu().numpy().view(np.uint32) == s_c.view(np.uint32), axis=1))
    assert rows.size >= 48
    q2, s2 = fp8bs.quantize_act(to_dev_bf16(y[rows]))
    assert torch.equal(q[rows].cpu(), q2.cpu()) and torch.equal(s[rows].cpu(), s2.cpu())


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
def test_norm_quant_full_size_sampled(kind):
    # [16384, 7168] as benchmarked (0.5% outlier channels x100); rows are
    # independent, so a seeded sample of 256 rows is compared exactly.
    n = wl.norm(16384, 7168, seed=0, with_beta=kind == orc.NORM_LAYER)
    q, s, mean, rstd = run_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6)
    rows = np.sort(np.random.default_rng(1).choice(16384, 256, replace=False))
    rows = np.concatenate([[0, 1, 16382, 16383], rows])
    check_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6, q, s, mean, rstd, rows=rows)


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
@pytest.mark.parametrize("K", [7168, 8192])
def test_norm_quant_beta_long_rows(kind, K):
    # Rows of 7168 / 8192 with beta run a separate instantiation; 3700 rows
    # are more than one pass of the grid, so warps take several rows each.
    n = wl.norm(3700, K, seed=K + kind, with_beta=True)
    q, s, mean, rstd = run_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6)
    rows = np.sort(np.random.default_rng(K).choice(3700, 96, replace=False))
    rows = np.concatenate([[0, 1, 3551, 3552, 3698, 3699], rows])
    check_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6, q, s, mean, rstd, rows=rows)


def _random_norm_cases(n=16, seed=31):
    """Seeded rows: lengths across the specialised, generic and CTA-per-row
    paths, both norm kinds, beta or none, a few eps values, padded strides."""
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        K = 128 * int(rng.choice([1, 3, 8, 16, 27, 56, 64, 90, 128, 200]))
        M = int(rng.integers(1, 40)) if K <= 16384 else int(rng.integers(1, 4))
        kind = [orc.NORM_RMS, orc.NORM_LAYER][i % 2]
        beta = bool(rng.random() < 0.5)
        eps = float(rng.choice([1e-6, 1e-5, 1e-3]))
        ldx = K + 8 * int(rng.choice([0, 0, 1, 5]))
        ldq = K + 16 * int(rng.choice([0, 0, 1, 3]))
        cases.append((M, K, kind, beta, eps, ldx, ldq))
    return cases


@pytest.mark.parametrize("M,K,kind,beta,eps,ldx,ldq", _random_norm_cases())
def test_norm_quant_random(M, K, kind, beta, eps, ldx, ldq):
    n = wl.norm(M, K, seed=M * 13 + K + kind, with_beta=beta)
    q, s, mean, rstd = run_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, eps, ldx=ldx, ldq=ldq)
    check_norm(n.x_bits, n.gamma_bits, n.beta_bits, kind, eps, q, s, mean, rstd)
