"""Pins for the oracle's NVFP4 -> bf16 dequantization, y = bf16_rn(fl32(S * dec(q)
* dec(s_b))) ("TRIAGE", section "NVFP4 quantization format and W4A4 execution";
the reading of the binary32 evaluation order is the one stated in the header).

Pinned by: hand-worked values (tests/golden/dequant_examples.txt), the exact
binary64 value of the same product (one bf16 rounding away, except where the
binary32 product lands on a bf16 tie), the round trip through the quantizer, and
the per-tensor (single scale) form.
"""
import os

import numpy as np
import pytest

from nvfp4_precision_rl_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant_examples.txt")


def _golden():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        s, sb, code, want = [f.strip() for f in line.split("|")]
        out.append((float.fromhex(s), int(sb, 16), int(code, 16), int(want, 16)))
    return out


def test_golden_examples(orc):
    cases = _golden()
    assert len(cases) >= 15
    for S, sb, code, want in cases:
        # one 16-element block holding the code in every position
        q = np.full((1, 8), code | (code << 4), np.uint8)
        sf = np.full((1, 1), sb, np.uint8)
        got = orc.dequantize_bf16(q, sf, np.array([S], np.float32))
        assert np.all(got == want), (S, hex(sb), code, hex(int(got[0, 0])), hex(want))


def _bf16_value(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_one_rounding_from_the_exact_product(orc):
    x = W.small_matrix(31, 96, 512, dist="student_t3", outlier_cols=3, outlier_scale=40)
    r = orc.quantize(x)
    exact = orc.dequantize(r["q"], r["sf"], r["s"])          # binary64, exact
    got = orc.dequantize_bf16(r["q"], r["sf"], r["s"])
    direct = orc.bf16_from_double(exact).reshape(exact.shape)
    val = _bf16_value(got)
    # within one bf16 rounding of the exact value (half an ulp, plus the binary32 step)
    ulp = np.maximum(np.abs(exact), 2.0 ** -133) * 2.0 ** -7
    assert np.all(np.abs(val - exact) <= 0.5 * ulp + np.abs(exact) * 2.0 ** -24)
    # equal to the single rounding except where fl32(p) is exactly a bf16 midpoint
    p32 = exact.astype(np.float32)
    tie = (p32.view(np.uint32) & 0xFFFF) == 0x8000
    assert np.array_equal(got[~tie], direct[~tie])
    assert np.all(np.sign(val) * np.sign(exact) >= 0)


def test_round_trip_error_bound(orc):
    """|dequant(quant(x)) - x| <= half an E2M1 step of the block (the largest
    step is 2: between 4 and 6) times dec(s_b) * S, plus the bf16 rounding."""
    x = W.small_matrix(32, 64, 1024)
    xf = W.bf16_bits_to_float(x).astype(np.float64)
    r = orc.quantize(x)
    y = _bf16_value(orc.dequantize_bf16(r["q"], r["sf"], r["s"]))
    dec_sf = orc.e4m3_table()[r["sf"]].astype(np.float64)          # [rows, K/16]
    step = np.repeat(dec_sf, 16, axis=1) * r["s"].astype(np.float64)[:, None]
    assert np.all(np.abs(y - xf) <= 1.0 * step + np.abs(xf) * 2.0 ** -8 + 1e-30)


def test_single_scale_form(orc):
    x = W.small_matrix(33, 40, 256)
    r = orc.quantize(x, mode="per_tensor")
    a = orc.dequantize_bf16(r["q"], r["sf"], r["s"], s_per_row=True)
    b = orc.dequantize_bf16(r["q"], r["sf"], r["s"][:1], s_per_row=False)
    assert np.array_equal(a, b)


def test_zero_codes_and_zero_scale(orc):
    q = np.zeros((3, 16), np.uint8)
    sf = np.full((3, 2), 0x38, np.uint8)
    assert not orc.dequantize_bf16(q, sf, np.ones(3, np.float32)).any()
    q = np.full((3, 16), 0x77, np.uint8)
    assert not orc.dequantize_bf16(q, sf, np.zeros(3, np.float32)).any()


def test_nibble_order_and_block_index(orc):
    """Low nibble = even element; block b's scale applies to elements 16b..16b+15."""
    q = np.zeros((1, 16), np.uint8)
    q[0, 0] = 0x71          # element 0: code 1 (0.5), element 1: code 7 (6)
    q[0, 8] = 0x0a          # element 16: code 0xa (-1)
    sf = np.array([[0x38, 0x40]], np.uint8)    # block 0: 1.0, block 1: 2.0
    got = orc.dequantize_bf16(q, sf, np.array([1.0], np.float32))
    assert got[0, 0] == 0x3f00 and got[0, 1] == 0x40c0 and got[0, 16] == 0xc000
    assert not got[0, 2:16].any() and not got[0, 17:].any()
