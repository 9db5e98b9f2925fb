"""Pins for the oracle's 1x128 activation and 128x128 weight quantizers.

Independent checks: hand-computed tiles with known amax, numpy's binary32
division plus a brute-force nearest-code search, the error bound of the
two roundings, and the outlier-containment property of fine grouping."""
import math

import numpy as np
import pytest

from fp8_fine_grained_17_b300 import workloads as wl


def _bits(vals):
    return wl.bf16_bits(np.asarray(vals, dtype=np.float32))


def _nearest_codes(table, y):
    """Vectorised nearest-even search over the finite codes, saturating."""
    finite = np.array([c for c in range(256) if not math.isnan(table[c])])
    vals = table[finite]
    out = np.empty(y.shape, dtype=np.uint8)
    for i, v in enumerate(y.ravel()):
        v = float(v)
        if v >= 448.0:
            out.flat[i] = 0x7E
            continue
        if v <= -448.0:
            out.flat[i] = 0xFE
            continue
        d = np.abs(vals - v)
        cand = finite[d == d.min()]
        if len(cand) > 1:
            cand = cand[(cand & 1) == 0]
        c = int(cand[0])
        if table[c] == 0.0:
            c = 0x80 if math.copysign(1.0, v) < 0 else 0x00
        out.flat[i] = c
    return out


def test_amax_448_is_identity(orc):
    table = orc.e4m3_table()
    codes = np.arange(0, 127, dtype=np.uint8)         # all non-negative finite codes
    vals = np.concatenate([table[codes], [448.0]])     # 128 values, amax 448
    x = _bits(vals)[None, :]
    q, s = orc.quantize_act_1x128(x)
    assert s[0, 0] == np.float32(1.0)
    assert np.array_equal(q[0, :127], codes)
    assert q[0, 127] == 0x7E


def test_zero_group(orc):
    x = _bits(np.zeros(256, dtype=np.float32))[None, :]
    x[0, 5] = 0x8000                                  # bf16 -0.0
    q, s = orc.quantize_act_1x128(x)
    assert np.all(s == 1.0)
    assert q[0, 5] == 0x80
    q[0, 5] = 0
    assert np.all(q == 0)


def test_amax_one(orc):
    vals = np.zeros(128, dtype=np.float32)
    vals[0], vals[1], vals[2] = 1.0, -1.0, 0.5
    q, s = orc.quantize_act_1x128(_bits(vals)[None, :])
    assert s[0, 0] == np.float32(1.0) / np.float32(448.0)
    assert q[0, 0] == 0x7E and q[0, 1] == 0xFE
    assert q[0, 2] == 0x76                             # 0.5/s = 224 exactly representable


def test_independent_restatement(orc):
    """numpy binary32 division + brute-force nearest code, per group."""
    table = orc.e4m3_table()
    rng = np.random.default_rng(3)
    M, K = 6, 384
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(3)
    x[1] *= np.float32(1e-30)
    x[2, :128] = 0
    x[3, 130] = np.float32(-7e4)
    xb = wl.bf16_bits(x)
    xf = wl.bits_to_f32(xb)
    q, s = orc.quantize_act_1x128(xb)
    for m in range(M):
        for g in range(K // 128):
            grp = xf[m, g * 128:(g + 1) * 128]
            amax = np.float32(np.max(np.abs(grp)))
            se = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(448.0))
            assert s[m, g] == se
            y = (grp / se).astype(np.float32)
            assert np.array_equal(q[m, g * 128:(g + 1) * 128], _nearest_codes(table, y))


def test_error_bound_and_amax_code(orc):
    """Each dequantized value is within half an E4M3 step (plus the binary32
    division's half ulp) of x, and the amax element always maps to +-448."""
    table = orc.e4m3_table()
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 512)).astype(np.float32) * np.float32(10) ** rng.integers(-20, 20, (64, 1)).astype(np.float32)
    xb = wl.bf16_bits(x)
    xf = wl.bits_to_f32(xb).astype(np.float64)
    q, s = orc.quantize_act_1x128(xb)
    sf = np.repeat(s.astype(np.float64), 128, axis=1)
    y = xf / sf
    deq = table[q]
    ay = np.abs(y)
    e = np.floor(np.log2(np.maximum(ay, 2.0 ** -6)))
    half_step = 2.0 ** (e - 4)
    assert np.all(np.abs(deq - y) <= half_step + ay * 2.0 ** -23)
    for m in range(64):
        for g in range(4):
            grp = xf[m, g * 128:(g + 1) * 128]
            i = int(np.argmax(np.abs(grp)))
            assert q[m, g * 128 + i] in (0x7E, 0xFE)


def test_outlier_containment(orc):
    """An outlier sets its own tile's scale and leaves its neighbours alone
    (fine-grained grouping accommodates outliers: "How Google Is Changing How
    We Method Deepseek", paragraph on adapting the scale to smaller groups)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 256)).astype(np.float32)
    x[0, 17] = np.float32(1e5) * np.float32(np.abs(x[0]).max())   # pushes the rest below E4M3 range
    xb = wl.bf16_bits(x)
    xf = wl.bits_to_f32(xb)
    q, s = orc.quantize_act_1x128(xb)
    assert s[0, 0] == np.float32(np.abs(xf[0, :128]).max() / np.float32(448.0))
    assert s[0, 1] == np.float32(np.abs(xf[0, 128:]).max() / np.float32(448.0))
    # the other elements of the outlier's tile lose resolution; the next tile does not
    table = orc.e4m3_table()
    deq = table[q[0]] * np.repeat(s[0].astype(np.float64), 128)
    rel = np.abs(deq - xf[0]) / np.abs(xf[0])
    others = np.ones(128, dtype=bool)
    others[17] = False
    assert np.mean(rel[:128][others]) > 2 * np.mean(rel[128:])
    assert np.count_nonzero((q[0, :128] & 0x7F) == 0) > 10      # flushed to +-0
    assert np.count_nonzero((q[0, 128:] & 0x7F) == 0) == 0
    # row 1 is untouched by row 0's outlier
    q1, s1 = orc.quantize_act_1x128(xb[1:2])
    assert np.array_equal(q1, q[1:2]) and np.array_equal(s1, s[1:2])


def test_weight_blocks(orc):
    rng = np.random.default_rng(6)
    N, K = 300, 256                                    # partial last row block
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[260, 3] = 5.0                                    # lives in the partial block (2, 0)
    wb = wl.bf16_bits(w)
    wf = wl.bits_to_f32(wb)
    q, s = orc.quantize_weight_128x128(wb)
    assert s.shape == (3, 2)
    for nb in range(3):
        for kb in range(2):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.float32(np.abs(blk).max())
            assert s[nb, kb] == np.float32(amax / np.float32(448.0))
            for n in range(nb * 128, min(N, nb * 128 + 128), 37):
                for k in range(kb * 128, kb * 128 + 128, 11):
                    assert q[n, k] == orc.quantize_value(wf[n, k], s[nb, kb])
    assert q[260, 3] == 0x7E


def test_act_equals_weight_quantizer_on_single_rows(orc):
    """A 1-row weight block has the same amax as a 1x128 tile."""
    rng = np.random.default_rng(7)
    x = wl.bf16_bits(rng.standard_normal((1, 512)).astype(np.float32))
    qa, sa = orc.quantize_act_1x128(x)
    qw, sw = orc.quantize_weight_128x128(x)
    assert np.array_equal(qa, qw) and np.array_equal(sa, sw)


def test_pairs_match_groups(orc):
    rng = np.random.default_rng(8)
    x = wl.bf16_bits(rng.standard_normal((3, 128)).astype(np.float32))
    q, s = orc.quantize_act_1x128(x)
    xf = wl.bits_to_f32(x)
    amax = wl.bf16_bits(np.abs(xf).max(axis=1, keepdims=True).repeat(128, axis=1))
    qp, sp = orc.quantize_pairs(amax, x)
    assert np.array_equal(qp.reshape(3, 128), q)
    assert np.array_equal(sp.reshape(3, 128)[:, 0], s[:, 0])


# ---------------------------------------------------------------- power-of-two scales

@pytest.mark.parametrize("amax,want", [
    (0.0, 1.0),              # all-zero group: s = 1
    (448.0, 1.0),            # 448 / 1 = 448 is allowed
    (449.0, 2.0),            # 449 / 1 > 448, 449 / 2 <= 448
    (1.0, 2.0 ** -8),        # 1 / 2^-8 = 256 <= 448 < 512
    (896.0, 2.0),
    (897.0, 4.0),
    (1.75, 2.0 ** -8),       # 1.75 * 256 = 448 exactly
    (1.7578125, 2.0 ** -7),  # next bf16 above 1.75: 450 > 448
])
def test_pow2_scale_hand_values(orc, amax, want):
    assert orc.group_scale_pow2(amax) == np.float32(want)


def test_pow2_scale_every_bf16_amax(orc):
    """For every positive finite bf16 amax: s is a power of two in
    [2^-127, 2^127], amax / s <= 448, and s / 2 would exceed 448 unless s is
    already the smallest allowed power (exact rational arithmetic)."""
    bits = np.arange(1, 0x7F80, dtype=np.uint16)
    amax = wl.bits_to_f32(bits).astype(np.float64)
    s = np.array([orc.group_scale_pow2(a) for a in amax], dtype=np.float64)
    mant, ex = np.frexp(s)
    assert np.all(mant == 0.5)                      # exact powers of two
    assert np.all((ex - 1 >= -127) & (ex - 1 <= 127))
    assert np.all(amax <= 448.0 * s)                 # exact: s is 2^e, 448 = 7 * 2^6
    smaller_ok = (ex - 1 > -127)
    assert np.all(amax[smaller_ok] > 448.0 * (s[smaller_ok] / 2))


def test_pow2_codes_are_nearest_grid(orc):
    """With s = 2^e, x / s is exact, so every code is the nearest E4M3 value of
    x / s (ties to even, saturating) -- checked by brute force on the grid."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((16, 256)) * np.exp(rng.uniform(-20, 20, (16, 1)))).astype(np.float32)
    xb = wl.bf16_bits(x)
    q, s = orc.quantize_act_1x128(xb, pow2=True)
    table = orc.e4m3_table()
    y = wl.bits_to_f32(xb).astype(np.float64) / np.repeat(s.astype(np.float64), 128, axis=1)
    assert np.array_equal(q, _nearest_codes(table, y))
    # The largest magnitude of each group has x / s in (224, 448], so its code
    # (rounded to the E4M3 grid, spacing 16 in [128, 256)) is in [224, 448].
    amax_code = np.abs(table[q]).reshape(16, 2, 128).max(axis=2)
    assert np.all((amax_code >= 224.0) & (amax_code <= 448.0))


def test_pow2_weight_blocks_match_single_groups(orc):
    rng = np.random.default_rng(22)
    w = wl.weights(rng, 200, 256)
    q, s = orc.quantize_weight_128x128(w, pow2=True)
    for nb in range(2):
        rows = slice(128 * nb, min(128 * nb + 128, 200))
        for kb in range(2):
            blk = wl.bits_to_f32(w[rows, 128 * kb:128 * kb + 128])
            assert s[nb, kb] == orc.group_scale_pow2(float(np.abs(blk).max()))
