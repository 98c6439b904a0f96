"""Pins for the oracle's W4A4 GEMM: Y = S_x[m] S_w[n] sum_k dec(q_x)dec(s_x)dec(q_w)dec(s_w)
("TRIAGE", section "NVFP4 quantization format and W4A4 execution": both operands
are NVFP4 and the tensor cores consume them natively; "Towards Blackwell-Native
8-bit and 4-bit RL", results item 10: the per-token FP32 scale belongs in the
GEMM epilogue).

The exact integer sum is checked against brute force in rational arithmetic, an
integer special case, float64 BLAS on the decoded operands, and the oracle's own
plain float64 loop.
"""
from fractions import Fraction

import numpy as np
import torch

from nvfp4_precision_rl_gb300 import workloads as W


def _rand_operand(rng, rows, K, sf_choices=None):
    q = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    if sf_choices is None:
        sf = rng.integers(0, 0x7F, size=(rows, K // 16), dtype=np.uint8)   # finite E4M3
    else:
        sf = rng.choice(np.array(sf_choices, np.uint8), size=(rows, K // 16))
    s = (rng.standard_normal(rows) * 0.01).astype(np.float32)
    return dict(q=q, sf=sf, s=s)


def _frac_value(code, table):
    return Fraction(float(table[code]))


def test_brute_force_tiny_shapes(orc):
    e2 = orc.e2m1_table()
    e4 = orc.e4m3_table()
    rng = np.random.default_rng(61)
    for M, N in [(1, 1), (2, 3), (4, 4)]:
        K = 64
        a, b = _rand_operand(rng, M, K), _rand_operand(rng, N, K)
        y = orc.gemm_exact(a, b)
        for m in range(M):
            for n in range(N):
                acc = Fraction(0)
                for k in range(K):
                    ca = (a["q"][m, k // 2] >> (4 * (k & 1))) & 15
                    cb = (b["q"][n, k // 2] >> (4 * (k & 1))) & 15
                    acc += (_frac_value(ca, e2) * _frac_value(a["sf"][m, k // 16], e4)
                            * _frac_value(cb, e2) * _frac_value(b["sf"][n, k // 16], e4))
                want = float(acc * Fraction(float(a["s"][m])) * Fraction(float(b["s"][n])))
                assert y[m, n] == want


def test_integer_special_case(orc):
    """All scales 1 (S = 1, s_b = 1.0 = code 0x38) and codes in {0, +1, -1}:
    the product is an integer matmul."""
    rng = np.random.default_rng(62)
    M, N, K = 37, 29, 256
    ia = rng.choice([0, 1, -1], size=(M, K))
    ib = rng.choice([0, 1, -1], size=(N, K))
    code = {0: 0, 1: 2, -1: 10}

    def pack(iv):
        c = np.vectorize(code.get)(iv).astype(np.uint8)
        return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)

    a = dict(q=pack(ia), sf=np.full((M, K // 16), 0x38, np.uint8), s=np.ones(M, np.float32))
    b = dict(q=pack(ib), sf=np.full((N, K // 16), 0x38, np.uint8), s=np.ones(N, np.float32))
    assert np.array_equal(orc.gemm_exact(a, b), (ia @ ib.T).astype(np.float64))


def test_exact_vs_float64_blas_and_loop(orc):
    x = W.small_matrix(63, 150, 512, outlier_cols=2)
    w = W.small_matrix(64, 70, 512, std=0.02)
    a, b = orc.quantize(x), orc.quantize(w)
    y, absy = orc.gemm_exact(a, b, with_abs=True)
    xa = torch.from_numpy(orc.dequantize(a["q"], a["sf"], a["s"]))
    xb = torch.from_numpy(orc.dequantize(b["q"], b["sf"], b["s"]))
    blas = (xa @ xb.T).numpy()
    loop = orc.gemm_fp64(a, b)
    for other in (blas, loop):
        assert np.all(np.abs(y - other) <= 1e-12 * absy + 1e-300)
    assert np.all(absy >= np.abs(y))


def test_sampled_matches_full(orc):
    x = W.small_matrix(65, 64, 256)
    w = W.small_matrix(66, 48, 256, std=0.02)
    a, b = orc.quantize(x), orc.quantize(w)
    y = orc.gemm_exact(a, b)
    rng = np.random.default_rng(0)
    mi = rng.integers(0, 64, 500)
    ni = rng.integers(0, 48, 500)
    ys, _ = orc.gemm_exact_sampled(a, b, mi, ni)
    assert np.array_equal(ys, y[mi, ni])


def test_quantization_error_is_small_for_gaussian_data(orc):
    """Sanity of the whole recipe: the W4A4 product tracks the bf16 product to
    the few-percent level expected of 4-bit operands."""
    x = W.small_matrix(67, 64, 1024)
    w = W.small_matrix(68, 64, 1024, std=0.02)
    y = orc.gemm_exact(orc.quantize(x), orc.quantize(w))
    ref = W.bf16_bits_to_float(x).astype(np.float64) @ W.bf16_bits_to_float(w).astype(np.float64).T
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert 0.01 < rel < 0.2
