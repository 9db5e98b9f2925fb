"""Pins for the oracle's normalization fused with the 1x128 cast.

Independent checks: PyTorch's float64 layer-norm and RMS-norm routines
(statistics and outputs), PyTorch's float32 -> bf16 conversion, closed forms
for rows whose statistics are known exactly, and scale invariance."""
import math

import numpy as np
import pytest
import torch

from fp8_fine_grained_17_b300 import workloads as wl
from oracle import oracle as orc

U32 = 2.0 ** -24   # unit roundoff of binary32


def _rows(M, K, seed, outliers=None, beta=True):
    rng = np.random.default_rng(seed)
    x, _ = wl.activations(rng, M, K, outliers)
    g, b = wl.norm_params(rng, K, beta)
    return x, g, b


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # Exact halfway cases (low 16 bits = 0x8000) with both parities, and their neighbours.
    base = rng.integers(0x0100, 0x7F00, 2000, dtype=np.uint32)   # finite, normal
    halves = ((base << 16) | 0x8000).view(np.float32)
    near = np.concatenate([halves, np.nextafter(halves, np.float32(np.inf)),
                           np.nextafter(halves, np.float32(-np.inf)), -halves])
    allv = np.concatenate([v, near, np.float32([0.0, -0.0, 1e-40, -1e-40])])
    assert np.array_equal(orc.f32_to_bf16_bits(allv), wl.bf16_bits(allv))


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
@pytest.mark.parametrize("K", [128, 384, 7168])
def test_stats_match_torch_float64(kind, K):
    x, _, _ = _rows(64, K, seed=K + kind, outliers=100.0)
    eps = 1e-6
    mu, rstd = orc.norm_stats(x, kind, eps)
    xt = torch.from_numpy(orc.bf16_bits_to_f32(x).astype(np.float64))
    if kind == orc.NORM_LAYER:
        _, m_t, r_t = torch.ops.aten.native_layer_norm(xt, [K], None, None, float(np.float32(eps)))
        m_ref = m_t[:, 0].numpy()
        # Same rounding argument as for rstd below; float64 summation order
        # adds at most ~1e-13 of the mean magnitude.
        slack = 2 * U32 * np.abs(m_ref) + 1e-13 * np.abs(xt.numpy()).mean(axis=1)
        assert np.all(np.abs(mu.astype(np.float64) - m_ref) <= slack)
    else:
        _, r_t = torch.ops.aten._fused_rms_norm(xt, [K], None, float(np.float32(eps)))
        assert np.all(mu == 0)
    r_ref = r_t[:, 0].numpy()
    # Both are float64 computations rounded once to binary32: at most one
    # binary32 ulp apart (a difference only when the float64 values straddle
    # a rounding boundary).
    rel = np.abs(rstd.astype(np.float64) - r_ref) / r_ref
    assert rel.max() <= 2 * U32 * 1.0001


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
@pytest.mark.parametrize("beta", [False, True])
def test_outputs_match_torch_float64(kind, beta):
    M, K = 48, 1024
    x, g, b = _rows(M, K, seed=7 + kind, outliers=50.0, beta=beta)
    eps = 1e-5
    _, _, mu, rstd, y = orc.norm_quantize_act_1x128(x, g, b, kind, eps)
    xt = torch.from_numpy(orc.bf16_bits_to_f32(x).astype(np.float64))
    gt = torch.from_numpy(orc.bf16_bits_to_f32(g).astype(np.float64))
    bt = torch.from_numpy(orc.bf16_bits_to_f32(b).astype(np.float64)) if beta else None
    e32 = float(np.float32(eps))
    if kind == orc.NORM_LAYER:
        ref = torch.nn.functional.layer_norm(xt, [K], gt, bt, e32)
    else:
        ref = torch.nn.functional.rms_norm(xt, [K], gt, e32)
        if bt is not None:
            ref = ref + bt
    ref = ref.numpy()
    got = orc.bf16_bits_to_f32(y).astype(np.float64)
    # bf16 rounding: half an ulp <= 2^-8 |v|; binary32 steps (rounded
    # statistics, subtract, two multiplies, add): a few u of the terms.
    xs = np.abs(orc.bf16_bits_to_f32(x).astype(np.float64))
    terms = (xs + np.abs(mu.astype(np.float64))[:, None]) * rstd[:, None] * np.abs(gt.numpy())[None, :]
    bound = 2.0 ** -8 * np.abs(ref) * (1 + 2.0 ** -7) + 8 * U32 * (terms + np.abs(ref)) + 1e-30
    assert np.all(np.abs(got - ref) <= bound)


def test_rms_closed_form():
    # Rows of +-c: mean(x^2) = c^2, so rstd = 1/sqrt(c^2 + eps) and, with
    # gamma = 1 and eps = 0, y = +-1 exactly; the 1x128 quantizer then maps
    # amax 1 to s = 1/448 and every code to +-448 (0x7E / 0xFE).
    K = 512
    rng = np.random.default_rng(3)
    c = np.float32([0.25, 3.0, 96.0, 2.0 ** -20])
    signs = np.where(rng.random((4, K)) < 0.5, -1.0, 1.0).astype(np.float32)
    x = wl.bf16_bits(signs * c[:, None])
    g = wl.bf16_bits(np.ones(K, np.float32))
    q, s, mu, rstd, y = orc.norm_quantize_act_1x128(x, g, None, orc.NORM_RMS, 0.0)
    assert np.array_equal(rstd, (1.0 / c.astype(np.float64)).astype(np.float32))
    assert np.array_equal(orc.bf16_bits_to_f32(y), signs)
    assert np.all(s == np.float32(1.0) / np.float32(448.0))
    assert np.array_equal(q, np.where(signs < 0, 0xFE, 0x7E).astype(np.uint8))
    # With eps the statistic is 1/sqrt(c^2 + eps) (float64, rounded once).
    eps = 0.5
    _, _, _, rstd_e, _ = orc.norm_quantize_act_1x128(x, g, None, orc.NORM_RMS, eps)
    want = np.float32([1.0 / math.sqrt(float(v) ** 2 + eps) for v in c])
    assert np.array_equal(rstd_e, want)


def test_layer_closed_form():
    # Rows b + a*(+-1) with as many + as -: mu = b, var = a^2 exactly, so
    # with eps = 0 the normalized value is +-1, then gamma and beta apply.
    K = 256
    rng = np.random.default_rng(4)
    signs = np.tile(np.float32([1.0, -1.0]), (3, K // 2))
    for r in range(3):
        rng.shuffle(signs[r])
    a = np.float32([0.5, 4.0, 1.0])
    b = np.float32([3.0, -64.0, 0.0])
    x = wl.bf16_bits(b[:, None] + a[:, None] * signs)
    g = wl.bf16_bits(np.full(K, 1.5, np.float32))
    be = wl.bf16_bits(np.full(K, 0.25, np.float32))
    _, _, mu, rstd, y = orc.norm_quantize_act_1x128(x, g, be, orc.NORM_LAYER, 0.0)
    assert np.array_equal(mu, b)
    assert np.array_equal(rstd, np.float32(1.0) / a)
    assert np.array_equal(orc.bf16_bits_to_f32(y), np.float32(1.5) * signs + np.float32(0.25))


def test_layer_constant_row_gives_beta():
    # A constant row has var 0: d = 0 exactly, so y = beta for any eps > 0.
    K = 384
    x = wl.bf16_bits(np.full((2, K), 7.5, np.float32))
    rng = np.random.default_rng(9)
    g, be = wl.norm_params(rng, K, True)
    q, s, mu, rstd, y = orc.norm_quantize_act_1x128(x, g, be, orc.NORM_LAYER, 1e-6)
    assert np.all(mu == np.float32(7.5))
    assert np.array_equal(y, np.stack([be, be]))
    q0, s0 = orc.quantize_act_1x128(np.stack([be, be]))
    assert np.array_equal(q, q0) and np.array_equal(s, s0)


@pytest.mark.parametrize("kind", [orc.NORM_RMS, orc.NORM_LAYER])
def test_power_of_two_scale_invariance(kind):
    # With eps = 0 both norms are invariant under x -> 2^j x, and scaling by a
    # power of two is exact in bf16 and binary32, so every output bit agrees.
    x, g, b = _rows(16, 640, seed=11, outliers=100.0)
    ref = orc.norm_quantize_act_1x128(x, g, b, kind, 0.0)
    for j in (-6, 5):
        xs = wl.bf16_bits(orc.bf16_bits_to_f32(x) * np.float32(2.0 ** j))
        got = orc.norm_quantize_act_1x128(xs, g, b, kind, 0.0)
        for a_, b_ in zip((ref[0], ref[1], ref[4]), (got[0], got[1], got[4])):
            assert np.array_equal(a_, b_)
        assert np.array_equal(got[3], ref[3] * np.float32(2.0 ** -j))


def test_f32_step_walks_representable_values():
    v = np.float32([1.0, -1.0, 0.0, 3.5e-3, -7.25e4, 2.0 ** -126])
    up = orc.f32_step(v, 1)
    down = orc.f32_step(v, -1)
    assert np.array_equal(up, np.nextafter(v, np.float32(np.inf)))
    assert np.array_equal(down, np.nextafter(v, np.float32(-np.inf)))
    # Several steps equal repeated nextafter, across a binade and through zero.
    w = np.float32(2.0)
    for _ in range(5):
        w = np.nextafter(w, np.float32(-np.inf))
    assert orc.f32_step(np.float32(2.0), -5) == w
    z = np.float32(0.0)
    for _ in range(3):
        z = np.nextafter(z, np.float32(-np.inf))
    assert orc.f32_step(np.float32(1e-45), -4) == z
    assert orc.f32_step(orc.f32_step(np.float32(0.3), 17), -17) == np.float32(0.3)


def test_stat_rings_cover_the_interval_once():
    # Every binary32 pair inside the interval appears in exactly one ring, the
    # oracle's own pair first; nothing outside the interval appears.
    mu, r = np.float32(0.0625), np.float32(1.5)
    mu_abs = 5 * float(np.spacing(mu))
    r_rel = 3 * float(np.spacing(r)) / float(r)
    seen = []
    rings = list(orc.norm_stat_rings(mu, r, orc.NORM_LAYER, mu_abs, r_rel, max_ring=50))
    assert rings[0][0] == 0 and rings[0][1][0] == mu and rings[0][2][0] == r
    for d, mus, rs in rings:
        seen += list(zip(mus.tolist(), rs.tolist()))
    # Brute force over a wide grid of neighbours, kept by value. 0.0625 is a
    # power of two: below it the spacing halves, so 10 steps fit there.
    want = set()
    for i in range(-40, 41):
        for j in range(-40, 41):
            m2, r2 = orc.f32_step(mu, i), orc.f32_step(r, j)
            if abs(float(m2) - float(mu)) <= mu_abs and abs(float(r2) - float(r)) <= r_rel * float(r):
                want.add((float(m2), float(r2)))
    assert len(want) == 16 * 7
    assert len(seen) == len(set(seen)) == len(want) and set(seen) == want
    assert rings[-1][0] == 10
    # RMSNorm: mu stays 0, rstd walks outward symmetrically.
    rms = list(orc.norm_stat_rings(0.0, r, orc.NORM_RMS, 0.0, r_rel, max_ring=50))
    assert [d for d, _, _ in rms] == [0, 1, 2, 3]
    assert all(np.all(m == 0) for _, m, _ in rms)


def test_rows_at_equals_full_path_at_central_statistics():
    # Evaluating a row under the oracle's own statistics through the candidate
    # path gives the rows of norm_quantize_act_1x128; a wrong rstd changes codes.
    for kind in (orc.NORM_RMS, orc.NORM_LAYER):
        x, g, b = _rows(6, 896, seed=21 + kind, outliers=100.0)
        q, s, mu, rstd, _ = orc.norm_quantize_act_1x128(x, g, b, kind, 1e-6)
        for i in range(6):
            qc, sc = orc.norm_rows_at(x[i], g, b, kind, mu[i:i + 1], rstd[i:i + 1])
            assert np.array_equal(qc[0], q[i]) and np.array_equal(sc[0], s[i])
        # A rstd about 25% larger scales y, hence every group's amax and
        # scale (the codes, being scale-free, mostly stay).
        far = orc.f32_step(rstd[:1], 1 << 21)
        assert 1.2 < far[0] / rstd[0] < 1.3
        _, sf = orc.norm_rows_at(x[0], g, b, kind, mu[:1], far)
        assert np.all(sf[0] != s[0])
