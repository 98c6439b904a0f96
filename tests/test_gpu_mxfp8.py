"""GPU parity of the MXFP8 quantizer and dequantizer against the oracle, bit-exact.

MXFP8: 32 values share one E8M0 power-of-two scale rounded up so the block
maximum fits E4M3's 448, the values E4M3 ("Towards Blackwell-Native 8-bit and
4-bit RL", MXFP8 format background); the 1x32 row copy and the 32x1 column
copy are quantized from the same bf16 data.  The GPU codes, the swizzled scale
bytes (padding included) and the dequantized bf16 must equal the oracle's.
Cases: ragged shapes (rows not a multiple of 128, K/32 not a multiple of 4),
random finite bf16 bit patterns over the whole exponent range (zero,
subnormal and near-overflow blocks), the column copy, a padded input pitch,
arbitrary code/scale bytes for the dequantizer, the Qwen3-4B up-projection
activation at full size, empty input and argument errors.
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import host, to_dev

pytestmark = pytest.mark.gpu


def _check(nv, orc, x_bits, column_copy=False, ld=None):
    rows, cols = x_bits.shape
    if ld is None:
        xd = to_dev(x_bits)
    else:
        full = np.full((rows, ld), 0x7F7F, np.uint16)   # finite junk in the gap
        full[:, :cols] = x_bits
        xd = to_dev(full)[:, :cols]
    got = nv.mxfp8_quantize(xd, column_copy=column_copy)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    want = orc.mxfp8_quantize(x_bits, column_copy=column_copy)
    for kg, kw in (("q", "q"), ("sf", "sf_swz")) + ((("q_col", "q_col"), ("sf_col", "sf_col_swz"))
                                                      if column_copy else ()):
        g, w = host(got[kg]).reshape(-1), want[kw].reshape(-1)
        assert g.shape == w.shape, kg
        bad = np.flatnonzero(g != w)
        assert bad.size == 0, f"{kg}: {bad.size} differ, first {bad[:5].tolist()}"
    return got, want


@pytest.mark.parametrize("M,K", [(1, 32), (7, 96), (130, 256), (257, 2080), (300, 2560), (64, 4128)])
def test_rows(nv, orc, M, K):
    _check(nv, orc, W.small_matrix(M * 5 + K, M, K, dist="student_t3", outlier_cols=min(3, K // 32)))


@pytest.mark.parametrize("M,K", [(32, 64), (96, 256), (160, 2080), (416, 2048)])
def test_column_copy(nv, orc, M, K):
    _check(nv, orc, W.small_matrix(M + 7 * K, M, K, dist="lognormal_rows", outlier_cols=2, outlier_scale=40),
           column_copy=True)


def test_all_exponents(nv, orc):
    """Random finite bf16 bit patterns: every block exponent, zero blocks,
    subnormals, values near the bf16 maximum."""
    rng = np.random.Generator(np.random.PCG64(77))
    x = rng.integers(0, 1 << 16, size=(192, 512), dtype=np.uint32).astype(np.uint16)
    x[(x & 0x7F80) == 0x7F80] &= 0xBFFF          # inf / NaN -> finite
    x[:32, :64] = 0                               # all-zero blocks (scale code 0)
    x[32:64, 64:128] &= 0x807F                    # subnormal-only blocks
    x[64:96, 128:160] = 0x8000                    # negative zeros
    _check(nv, orc, x, column_copy=True)


def test_padded_pitch(nv, orc):
    _check(nv, orc, W.small_matrix(9, 96, 320), column_copy=True, ld=328)


def test_dequantize(nv, orc):
    x = W.small_matrix(5, 200, 1056, dist="student_t3", outlier_cols=4)
    got, want = _check(nv, orc, x)
    y = nv.mxfp8_dequantize(got)
    torch.cuda.synchronize()
    assert np.array_equal(host(y), orc.mxfp8_dequantize_bf16(want["q"], want["sf"]))


def test_dequantize_column_copy(nv, orc):
    x = W.small_matrix(6, 128, 256, outlier_cols=2)
    got, want = _check(nv, orc, x, column_copy=True)
    y = nv.mxfp8_dequantize(got, column=True)
    torch.cuda.synchronize()
    assert np.array_equal(host(y), orc.mxfp8_dequantize_bf16(want["q_col"], want["sf_col"]))


def test_dequantize_arbitrary_bytes(nv, orc):
    """Every E4M3 code but NaN and every E8M0 code but NaN (255): products
    that underflow to bf16 subnormals and overflow to infinity included."""
    rng = np.random.Generator(np.random.PCG64(78))
    rows, cols = 136, 640
    q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint16).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] ^= 0x01
    sf = rng.integers(0, 255, size=(rows, cols // 32), dtype=np.uint16).astype(np.uint8)
    sf[0, :] = 0
    sf[1, :] = 254
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mxfp8_dequantize(torch.from_numpy(q).cuda(), torch.from_numpy(orc.sf_swizzle(sf)).cuda(), rows,
                              cols, y, cols)
    torch.cuda.synchronize()
    assert np.array_equal(host(y), orc.mxfp8_dequantize_bf16(q, sf))


def test_qwen3_4b_activation_full(nv, orc):
    _check(nv, orc, W.config2().x, column_copy=True)


def test_empty_and_errors(nv):
    x = torch.zeros((40, 64), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((64, 64), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    nv.nvfp4_mxfp8_quantize(x, 0, 64, 64, q, sf)                      # rows == 0: no-op
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_mxfp8_quantize(x, 40, 48, 64, q, sf)                 # cols % 32 != 0
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_mxfp8_quantize(x, 40, 64, 64, q, sf, q, sf)          # column copy needs rows % 32 == 0
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_mxfp8_quantize(x, 32, 64, 64, q, sf, q, None)        # q_col without sf_col
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_mxfp8_dequantize(q, sf, 4, 64, x, 60)                # ld_y < cols
    assert nv.nvfp4_mxfp8_sf_bytes(130, 2080) == 256 * 68
    assert nv.nvfp4_mxfp8_sf_bytes(0, 64) == 0
