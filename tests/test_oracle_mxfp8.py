"""Pins for the oracle's MXFP8 quantizer and dequantization ("Towards
Blackwell-Native 8-bit and 4-bit RL", "MXFP8 format background": 1x32 blocks,
E4M3 values, one E8M0 power-of-two scale rounded up so the block maximum is not
clipped; "Backward activation representation trade-off": the 1x32 row copy and
the 32x1 column copy are quantized independently from full precision).

Pinned by hand-worked blocks (tests/golden/mxfp8_examples.txt), the minimality
of the rounded-up scale, torch's float8_e4m3fn codec on x / 2^e, the exact
dequantization, and the column copy as the row copy of the transpose.
"""
import os

import numpy as np
import torch

from nvfp4_precision_rl_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp8_examples.txt")


def _bits(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _parse(tok):
    return float.fromhex(tok) if tok.startswith(("0x", "-0x")) else float(tok)


def test_golden_blocks(orc):
    n = 0
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        vals, code, codes = [f.split() for f in line.split("|")]
        v = [_parse(t) for t in vals]
        x = np.zeros((1, 32), np.uint16)
        x[0, :len(v)] = _bits(v)
        assert np.all(W.bf16_bits_to_float(x[0, :len(v)]) == np.array(v, np.float32)), "not bf16"
        r = orc.mxfp8_quantize(x)
        assert r["sf"][0, 0] == int(code[0], 16), (vals, hex(r["sf"][0, 0]))
        assert [int(c, 16) for c in codes] == list(r["q"][0, :len(v)]), (vals, [hex(c) for c in r["q"][0, :len(v)]])
        assert not r["q"][0, len(v):].any()
        n += 1
    assert n == 5


def test_scale_is_the_smallest_unclipped_power_of_two(orc):
    x = W.small_matrix(41, 64, 1024, dist="student_t3", outlier_cols=4, outlier_scale=1e3)
    r = orc.mxfp8_quantize(x)
    xf = np.abs(W.bf16_bits_to_float(x).astype(np.float64)).reshape(64, 32, 32)
    amax = xf.max(axis=2)
    e = r["sf"].astype(np.int64) - 127
    assert np.all(amax <= 448.0 * np.ldexp(1.0, e))
    assert np.all((e == -127) | (amax > 448.0 * np.ldexp(1.0, e - 1)))


def test_elements_match_torch_e4m3(orc):
    x = W.small_matrix(42, 96, 512, dist="lognormal_rows")
    r = orc.mxfp8_quantize(x)
    e = np.repeat(r["sf"].astype(np.int64) - 127, 32, axis=1)
    scaled = torch.from_numpy(np.ldexp(W.bf16_bits_to_float(x).astype(np.float64), -e).astype(np.float32))
    ref = scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(r["q"], ref)


def test_dequantize_exact_and_round_trip(orc):
    x = W.small_matrix(43, 64, 256)
    r = orc.mxfp8_quantize(x)
    y = orc.mxfp8_dequantize_bf16(r["q"], r["sf"])
    dec = torch.from_numpy(r["q"]).view(torch.float8_e4m3fn).double().numpy()
    e = np.repeat(r["sf"].astype(np.int64) - 127, 32, axis=1)
    exact = dec * np.ldexp(1.0, e)
    assert np.array_equal(W.bf16_bits_to_float(y).astype(np.float64), exact)   # 4 significant bits: exact
    xf = W.bf16_bits_to_float(x).astype(np.float64)
    # E4M3 relative step 2^-3 (half: 2^-4) above its smallest normal, absolute 2^-10 * 2^e below
    assert np.all(np.abs(exact - xf) <= np.abs(xf) * 2.0 ** -4 + np.ldexp(2.0 ** -10, e))


def test_column_copy_is_the_row_copy_of_the_transpose(orc):
    x = W.small_matrix(44, 96, 160)
    r = orc.mxfp8_quantize(x, column_copy=True)
    t = orc.mxfp8_quantize(np.ascontiguousarray(x.T))
    assert np.array_equal(r["q_col"], t["q"]) and np.array_equal(r["sf_col"], t["sf"])
