"""Pins for the oracle's two-level quantizer, swizzle and column-wise copy.

The decode contract is x ~ S * s_b * Q_E2M1(x / (S * s_b)) ("TRIAGE", section
"NVFP4 quantization format and W4A4 execution"), with a per-token FP32 outer
scale computed online ("Towards Blackwell-Native 8-bit and 4-bit RL", section
"Online per-token scale").  The checks: hand-worked examples, exact round trips
of representable rows, the nearest-value error bound, per-token batch
invariance (and its failure under a per-tensor scale), the pages' four test
classes (random / boundary / zeros / maxes), and layout positions.
"""
import os

import numpy as np
import pytest

from nvfp4_precision_rl_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_POS = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _codes(q):
    """packed [rows, K/2] -> codes [rows, K] (low nibble first)."""
    q = np.asarray(q, np.uint8)
    out = np.empty((q.shape[0], q.shape[1] * 2), np.uint8)
    out[:, 0::2] = q & 15
    out[:, 1::2] = q >> 4
    return out


def _signed_value(codes):
    mag = E2M1_POS[codes & 7]
    return np.where(codes & 8, -mag, mag)


def _num(s):
    return float.fromhex(s) if s.startswith(("0x", "-0x")) else float(s)


def test_golden_examples(orc):
    with open(os.path.join(GOLDEN, "quantize_examples.txt")) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert lines
    for ln in lines:
        xs, qs, sfs, ss = [p.split() for p in ln.split("|")]
        x = W.to_bf16_bits(np.array([_num(v) for v in xs], np.float32))[None, :]
        d = orc.quantize(x, nthreads=1)
        assert d["q"][0].tolist() == [int(b, 16) for b in qs]
        assert d["sf"][0].tolist() == [int(b, 16) for b in sfs]
        assert d["s"][0] == np.float32(_num(ss[0]))


def _representable_rows(rng, rows, K):
    """Rows x = S * sb_b * q with S a power of two, each block holding a +-6
    code, and one block with sb = 448 (so the row amax is 2688 * S)."""
    e4 = __import__("torch").arange(127, dtype=__import__("torch").uint8).view(
        __import__("torch").float8_e4m3fn).float().numpy()
    x = np.zeros((rows, K), np.float32)
    for r in range(rows):
        S = np.float32(2.0) ** int(rng.integers(-24, 12))
        sbs = rng.choice(e4[8:], size=K // 16)          # normal E4M3 values
        sbs[int(rng.integers(0, K // 16))] = 448.0
        for b in range(K // 16):
            q = rng.choice(np.concatenate([E2M1_POS, -E2M1_POS]), size=16)
            q[int(rng.integers(0, 16))] = 6.0 if rng.random() < 0.5 else -6.0
            x[r, 16 * b:16 * b + 16] = q * sbs[b] * S
    return x


def test_round_trip_of_representable_rows(orc):
    rng = np.random.default_rng(21)
    x = _representable_rows(rng, 64, 256)
    xb = W.to_bf16_bits(x)
    assert np.array_equal(W.bf16_bits_to_float(xb), x)       # exactly representable
    d = orc.quantize(xb)
    xhat = orc.dequantize(d["q"], d["sf"], d["s"])
    assert np.array_equal(xhat, x.astype(np.float64))
    # and re-quantizing the decoded row gives the same bytes
    d2 = orc.quantize(W.to_bf16_bits(xhat.astype(np.float32)))
    for key in ("q", "sf", "s"):
        assert np.array_equal(d[key], d2[key])


@pytest.mark.parametrize("dist", ["normal", "student_t3", "lognormal_rows"])
def test_nearest_value_error_bound(orc, dist):
    """Each element decodes to a nearest E2M1 grid point of x / (S * s_b) (up to
    the few-ulp FP32 error of forming that quotient), unless it saturates."""
    x = W.small_matrix(31, 96, 512, dist=dist, outlier_cols=3)
    d = orc.quantize(x)
    xf = W.bf16_bits_to_float(x).astype(np.float64)
    e4 = orc.e4m3_table()
    scale = d["s"].astype(np.float64)[:, None] * np.repeat(e4[d["sf"]], 16, axis=1)
    codes = _codes(d["q"])
    val = _signed_value(codes)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = np.where(scale > 0, xf / scale, 0.0)
    a = np.abs(y)
    gap = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    sat = a > 6.0
    err = np.abs(y - val)
    assert np.all(err[~sat] <= gap[~sat] / 2 + 4e-7 * a[~sat])
    assert np.all(np.abs(val[sat]) == 6.0)
    assert np.all(np.sign(val[val != 0]) == np.sign(y[val != 0]))


def test_scale_choice_puts_amax_block_at_448(orc):
    x = W.small_matrix(32, 200, 1024, dist="student_t3")
    d = orc.quantize(x)
    assert np.all(d["sf"].max(axis=1) == 0x7E)
    assert np.all((_codes(d["q"]) & 7).max(axis=1) == 7)
    amax = np.abs(W.bf16_bits_to_float(x)).max(axis=1)
    assert np.array_equal(d["s"], (amax / np.float32(2688.0)).astype(np.float32))


def test_per_token_batch_invariance(orc):
    """A token quantized alone equals the same token inside any batch
    ("Towards Blackwell-Native 8-bit and 4-bit RL", "Why per-token activation
    scaling": a shared scale makes a token's bytes depend on its batch)."""
    x = W.small_matrix(33, 160, 768, dist="student_t3", outlier_cols=8, outlier_scale=50)
    full = orc.quantize(x)
    rng = np.random.default_rng(3)
    for r in rng.choice(160, 12, replace=False):
        alone = orc.quantize(x[r:r + 1])
        assert np.array_equal(alone["q"][0], full["q"][r])
        assert np.array_equal(alone["sf"][0], full["sf"][r])
        assert alone["s"][0] == full["s"][r]
    sub = orc.quantize(x[40:90])
    assert np.array_equal(sub["q"], full["q"][40:90])


def test_per_tensor_scale_is_batch_dependent(orc):
    """The same check fails under a per-tensor outer scale on heavy-tailed rows."""
    x = W.small_matrix(34, 160, 768, dist="student_t3", outlier_cols=8, outlier_scale=50)
    full = orc.quantize(x, mode="per_tensor")
    assert np.all(full["s"] == full["s"][0])
    differs = 0
    for r in range(0, 160, 16):
        alone = orc.quantize(x[r:r + 1], mode="per_tensor")
        differs += not np.array_equal(alone["q"][0], full["q"][r])
    assert differs > 0


def test_zeros_class(orc):
    x = W.init_data_class("zeros", 41, 8, 128)
    d = orc.quantize(x)
    assert np.all(d["s"] == 0) and np.all(d["sf"] == 0)
    sign = (x >> 15).astype(np.uint8)
    assert np.array_equal(_codes(d["q"]), sign * 8)


def test_maxes_class(orc):
    x = W.init_data_class("maxes", 42, 8, 128)
    d = orc.quantize(x)
    assert np.all(d["sf"] == 0x7E)
    codes = _codes(d["q"])
    sign = (x >> 15).astype(np.uint8)
    assert np.array_equal(codes, 7 + 8 * sign)
    assert np.all(np.isfinite(d["s"]))


def test_boundary_class_ties(orc):
    """Blocks whose scaled elements sit exactly on E2M1 ties, or whose block
    scale sits exactly on an E4M3 tie, round to the even neighbour."""
    x = W.init_data_class("boundary", 43, 16, 256)
    d = orc.quantize(x)
    xf = W.bf16_bits_to_float(x).astype(np.float64)
    e4 = orc.e4m3_table()
    codes = _codes(d["q"])
    checked_e2m1 = checked_e4m3 = 0
    for r in range(x.shape[0]):
        S = float(d["s"][r])
        assert S == 2.0 ** np.round(np.log2(S))          # exact power of two
        for b in range(1, x.shape[1] // 16):
            blk = xf[r, 16 * b:16 * b + 16]
            dq = np.abs(blk).max() / (6 * S)              # exact: the block's E4M3 target
            lo = e4[:0x7F][e4[:0x7F] <= dq].max()
            i = int(np.where(e4[:0x7F] == lo)[0][0])
            if dq == lo and dq == 2.0 ** np.round(np.log2(dq)):
                assert d["sf"][r, b] == i
                y = blk / (S * dq)
                assert np.array_equal(codes[r, 16 * b:16 * b + 16], _e2m1_ref(y))
                checked_e2m1 += 1
            elif i + 1 < 0x7F and dq == (e4[i] + e4[i + 1]) / 2:
                assert d["sf"][r, b] == (i if i % 2 == 0 else i + 1)
                checked_e4m3 += 1
    assert checked_e2m1 > 20 and checked_e4m3 > 20


def _e2m1_ref(y):
    a = np.abs(y)
    v = np.where(a < 2.0, np.round(a * 2.0) / 2.0,
                 np.where(a < 4.0, np.round(a), 2.0 * np.round(a / 2.0)))
    code = np.searchsorted(E2M1_POS, np.minimum(v, 6.0))
    return (code + 8 * np.signbit(y)).astype(np.uint8)


def test_swizzle_golden_positions(orc):
    with open(os.path.join(GOLDEN, "sf_swizzle_positions.txt")) as f:
        rows = [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]
    R, KB = rows[0][0], rows[0][1]
    assert orc.sf_swizzled_bytes(R, KB) == 4608
    sf = np.zeros((R, KB), np.uint8)
    for _, _, r, c, off in rows:
        sf[:] = 0
        sf[r, c] = 0xAB
        swz = orc.sf_swizzle(sf)
        assert np.nonzero(swz)[0].tolist() == [off]


def test_swizzle_is_a_bijection(orc):
    rng = np.random.default_rng(5)
    for rows, kb in [(1, 1), (128, 4), (300, 10), (257, 33)]:
        sf = rng.integers(1, 255, size=(rows, kb), dtype=np.uint8)
        swz = orc.sf_swizzle(sf)
        assert swz.size == orc.sf_swizzled_bytes(rows, kb)
        assert np.count_nonzero(swz) == rows * kb        # pads stay zero, no collisions
        assert np.array_equal(orc.sf_unswizzle(swz, rows, kb), sf)


def test_column_copy(orc):
    """Column-wise copy: X^T quantized along tokens with one per-tensor scale
    from the global amax ("Towards Blackwell-Native 8-bit and 4-bit RL",
    "Backward activation representation": row- and column-wise copies are
    quantized independently from full precision)."""
    x = W.small_matrix(51, 96, 160, outlier_cols=2)
    d = orc.quantize(x, column_copy=True)
    xf = W.bf16_bits_to_float(x)
    amax = np.abs(xf).max()
    assert d["s_col"][0] == np.float32(amax) / np.float32(2688.0)
    # the same bytes as per-tensor row quantization of X^T
    t = orc.quantize(np.ascontiguousarray(x.T), mode="per_tensor")
    assert np.array_equal(d["q_col"], t["q"]) and np.array_equal(d["sf_col"], t["sf"])
    # decoded copy is within the per-block nearest-value bound of X^T
    xhat = orc.dequantize(d["q_col"], d["sf_col"], np.full(160, d["s_col"][0], np.float32))
    e4 = orc.e4m3_table()
    blk = d["s_col"][0] * np.repeat(e4[d["sf_col"]], 16, axis=1)
    assert np.all(np.abs(xhat - xf.T) <= blk * 1.0 + 1e-30)


def test_gather_rows(orc):
    x = W.small_matrix(52, 40, 64)
    g = np.array([3, -1, 39, 3, 0, -1], np.int32)
    d = orc.quantize(x, gather=g)
    full = orc.quantize(x)
    for i, src in enumerate(g):
        if src < 0:
            assert not d["q"][i].any() and not d["sf"][i].any() and d["s"][i] == 0
        else:
            assert np.array_equal(d["q"][i], full["q"][src])
            assert np.array_equal(d["sf"][i], full["sf"][src])
