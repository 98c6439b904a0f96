"""Pins for the oracle's element formats (E2M1 values, E4M3 block scales).

Each check compares the oracle with something outside it: the value set the
pages name for E2M1, torch's float8_e4m3fn codec, a banker's-rounding
formulation of E2M1 rounding, and hand-worked anchors under tests/golden/.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_e2m1_table_is_the_value_set(orc):
    t = orc.e2m1_table()
    for code, val in _rows("e2m1_values.txt"):
        v = float(val)
        assert t[int(code)] == v
        assert np.signbit(t[int(code)]) == np.signbit(v)


def test_e4m3_table_matches_torch_float8(orc):
    t = orc.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(t[~nan], ref[~nan])
    assert t[0x7E] == 448.0 and t[0x01] == 2.0 ** -9


def test_e2m1_golden_rounding(orc):
    rows = _rows("e2m1_rounding.txt")
    x = np.array([float(a) for a, _ in rows], np.float32)
    want = np.array([int(c) for _, c in rows], np.uint8)
    assert np.array_equal(orc.e2m1_encode(x), want)


def test_e4m3_golden_points(orc):
    rows = _rows("e4m3_points.txt")
    x = np.array([float(a) for a, _ in rows], np.float32)
    want = np.array([int(c, 16) for _, c in rows], np.uint8)
    assert np.array_equal(orc.e4m3_encode(x), want)


def _e2m1_bankers(x):
    """E2M1 rounding restated with numpy's round-half-even on each binade:
    spacing 0.5 below 2, 1 on [2, 4), 2 on [4, 6], saturating at 6."""
    a = np.abs(x.astype(np.float64))
    v = np.where(a < 2.0, np.round(a * 2.0) / 2.0,
                 np.where(a < 4.0, np.round(a), 2.0 * np.round(a / 2.0)))
    v = np.minimum(v, 6.0)
    # value -> code within the positive half of the table
    code = np.searchsorted(np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6]), v)
    return (code + 8 * np.signbit(x)).astype(np.uint8)


def test_e2m1_encoder_vs_bankers_rounding(orc):
    rng = np.random.default_rng(11)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    mids = (grid[1:] + grid[:-1]) / 2
    pts = np.concatenate([grid, mids, np.nextafter(mids.astype(np.float32), 0),
                          np.nextafter(mids.astype(np.float32), 10)]).astype(np.float32)
    rnd = rng.uniform(-8, 8, 200_000).astype(np.float32)
    x = np.concatenate([pts, -pts, rnd])
    assert np.array_equal(orc.e2m1_encode(x), _e2m1_bankers(x))


def test_e4m3_encoder_vs_torch_cast(orc):
    rng = np.random.default_rng(12)
    t = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = ((t[1:] + t[:-1]) / 2).astype(np.float32)      # every tie, exactly
    near = np.concatenate([np.nextafter(mids, 0), np.nextafter(mids, 1000)])
    logs = np.exp2(rng.uniform(-12, np.log2(464), 200_000)).astype(np.float32)
    x = np.concatenate([t.astype(np.float32), mids, near, logs])
    x = x[x <= 464]                                        # torch turns > 464 into NaN
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(x), ref)


def test_e4m3_saturates(orc):
    x = np.array([464.0, 465.0, 479.0, 480.0, 1e6, 3e38, np.inf], np.float32)
    assert np.all(orc.e4m3_encode(x) == 0x7E)


def test_decode_encode_round_trip(orc):
    e2 = orc.e2m1_table().astype(np.float32)
    assert np.array_equal(orc.e2m1_encode(e2), np.arange(16, dtype=np.uint8))
    e4 = orc.e4m3_table()[:0x7F].astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(e4), np.arange(0x7F, dtype=np.uint8))


def test_bf16_from_double_exact_rounding(orc):
    """bf16 rounding of binary64 values, against exact rational arithmetic."""
    from fractions import Fraction
    rng = np.random.default_rng(13)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8) * 2.0 ** 40,
                         1.0 + 2.0 ** -8 + 2.0 ** -40, 0.0, -0.0]])
    got = orc.bf16_from_double(v)

    def ref(x):
        if x == 0:
            return 0x8000 if np.signbit(x) else 0
        f = Fraction(abs(x))
        e = f.numerator.bit_length() - f.denominator.bit_length()
        while Fraction(2) ** e > f:
            e -= 1
        while Fraction(2) ** (e + 1) <= f:
            e += 1
        q = f / Fraction(2) ** (e - 7)          # in [128, 256)
        n = q.numerator // q.denominator
        rem = q - n
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
            n += 1
        val = float(Fraction(n) * Fraction(2) ** (e - 7))
        bits = int(np.array([val], np.float32).view(np.uint32)[0]) >> 16
        return bits | (0x8000 if x < 0 else 0)

    want = np.array([ref(x) for x in v], np.uint16)
    assert np.array_equal(got, want)
