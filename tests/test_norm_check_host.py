"""The fused-norm parity checker on the CPU.

Rows produced at a binary32 statistic a few ulps from the correctly rounded
one (as a parallel sum gives) must be accepted; a single wrong code or scale,
or statistics outside the proven interval, must be rejected."""
import numpy as np
import pytest

from fp8_fine_grained_17_b300 import workloads as wl
from oracle import oracle as orc

from helpers import check_norm_rows, norm_rstd_bound


def _case(kind, M=24, K=1024, seed=3):
    n = wl.norm(M, K, seed=seed, with_beta=kind == orc.NORM_LAYER)
    mu, r = orc.norm_stats(n.x_bits, kind, 1e-6)
    return n, mu, r


def _rows_at(n, kind, mu, r):
    q = np.empty(n.x_bits.shape, np.uint8)
    s = np.empty((n.x_bits.shape[0], n.x_bits.shape[1] // 128), np.float32)
    for i in range(n.x_bits.shape[0]):
        qi, si = orc.norm_rows_at(n.x_bits[i], n.gamma_bits, n.beta_bits, kind, mu[i:i + 1], r[i:i + 1])
        q[i], s[i] = qi[0], si[0]
    return q, s


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
def test_offcentre_statistics_accepted(kind):
    n, mu, r = _case(kind)
    rng = np.random.default_rng(0)
    r_k = orc.f32_step(r, rng.integers(-6, 7, r.size))
    mu_k = orc.f32_step(mu, rng.integers(-3, 4, mu.size)) if kind == orc.NORM_LAYER else mu
    q, s = _rows_at(n, kind, mu_k, r_k)
    rows, off, ring = check_norm_rows(orc, n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6, q, s, mu_k, r_k)
    assert rows == 24 and ring <= 6


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
def test_wrong_code_rejected(kind):
    n, mu, r = _case(kind)
    q, s = _rows_at(n, kind, mu, r)
    q[5, 300] ^= 1
    with pytest.raises(AssertionError, match="row 5"):
        check_norm_rows(orc, n.x_bits, n.gamma_bits, n.beta_bits, kind, 1e-6, q, s, mu, r, max_ring=8)


def test_wrong_scale_rejected():
    n, mu, r = _case(orc.NORM_RMS)
    q, s = _rows_at(n, orc.NORM_RMS, mu, r)
    s[2, 3] = np.nextafter(s[2, 3], np.float32(1))
    with pytest.raises(AssertionError, match="row 2"):
        check_norm_rows(orc, n.x_bits, n.gamma_bits, n.beta_bits, orc.NORM_RMS, 1e-6, q, s, mu, r, max_ring=8)


def test_statistic_outside_interval_rejected():
    n, mu, r = _case(orc.NORM_RMS)
    q, s = _rows_at(n, orc.NORM_RMS, mu, r)
    r_bad = r.copy()
    r_bad[0] = np.float32(r[0] * (1 + 2 * norm_rstd_bound(1024)))
    with pytest.raises(AssertionError, match="rstd off"):
        check_norm_rows(orc, n.x_bits, n.gamma_bits, n.beta_bits, orc.NORM_RMS, 1e-6, q, s, mu, r_bad)
