"""Pins for the oracle's E4M3 codec, against things other than itself:
hand-derived values from the format definition, brute-force nearest search
over the code table, and torch's float8_e4m3fn cast (a library routine)."""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_spot_values(orc):
    for code, val in _rows("e4m3_spot_values.txt"):
        got = orc.e4m3_decode(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val), (code, got, val)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val)), code


def test_rounding_cases(orc):
    for row in _rows("e4m3_rounding_cases.txt"):
        x, code = row[0], int(row[1], 16)
        assert orc.e4m3_encode(float(x)) == code, (x, hex(orc.e4m3_encode(float(x))), hex(code))


def test_all_codes_round_trip(orc):
    n_nan = 0
    for c in range(256):
        v = orc.e4m3_decode(c)
        if math.isnan(v):
            n_nan += 1
            assert c in (0x7F, 0xFF)
            continue
        assert orc.e4m3_encode(v) == c, hex(c)
    assert n_nan == 2


def test_decode_monotone_and_symmetric(orc):
    t = orc.e4m3_table()
    pos = t[0:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert pos[-1] == 448.0
    for c in range(0x7F):
        assert t[c | 0x80] == -t[c]


def test_matches_torch_cast_in_range(orc):
    # torch's float8_e4m3fn cast rounds to nearest even; inside +-448 it must agree.
    rng = np.random.default_rng(1)
    y = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(50),
        (rng.random(20000) * 2.0 ** rng.integers(-14, 9, 20000)).astype(np.float32),
        np.linspace(-448, 448, 4001, dtype=np.float32),
    ])
    y = y[np.abs(y) <= 448]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([orc.e4m3_encode(float(v)) for v in y], dtype=np.uint8)
    # torch maps results that round to zero to +0 or -0 by sign too
    assert np.array_equal(ours, ref)


def _brute_nearest(table, y):
    """Nearest finite code by scanning all codes; ties to the even code."""
    if y >= 448.0:
        return 0x7E
    if y <= -448.0:
        return 0xFE
    best = None
    for c in range(256):
        v = table[c]
        if math.isnan(v):
            continue
        d = abs(v - y)
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
        elif key == best[0]:
            # equal distance and parity: +0/-0 pair; keep the input's sign
            pass
    c = best[1]
    if table[c] == 0.0:
        return 0x80 if math.copysign(1.0, y) < 0 else 0x00
    return c


def test_brute_force_nearest(orc):
    table = orc.e4m3_table()
    finite = sorted(set(v for v in table if not math.isnan(v)))
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    cases = []
    for m in mids:
        f = np.float32(m)
        cases += [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    rng = np.random.default_rng(2)
    cases += list((rng.standard_normal(3000) * 100).astype(np.float32))
    cases += [np.float32(v) for v in (448.0, 449.0, 463.9, 464.0, 464.1, 480.0, 1e30, -1e30)]
    for y in cases:
        y = float(y)
        assert orc.e4m3_encode(y) == _brute_nearest(table, y), y
