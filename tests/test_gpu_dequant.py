"""GPU parity of nvfp4_dequantize (NVFP4 -> bf16) against the oracle, bit-exact.

Inputs are the oracle's own quantization of seeded bf16 data (codes, swizzled
scales, outer scales); the GPU result must equal orc.dequantize_bf16 bit for
bit.  Cases: ragged shapes (rows not a multiple of 128, K/16 not a multiple of
4), the column-wise copy with its single per-tensor scale, a padded output
pitch, empty input, the config-2 activation at full size, and argument errors.
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import host

pytestmark = pytest.mark.gpu


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda()


def _run(nv, q, sf_swz, s, per_row, rows, cols, ld=None):
    ld = cols if ld is None else ld
    y = torch.full((rows, ld), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    nv.nvfp4_dequantize(_dev(q), _dev(sf_swz), _dev(s), per_row, rows, cols, y, ld)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    return host(y)


@pytest.mark.parametrize("M,K", [(1, 16), (7, 48), (130, 256), (257, 2064), (300, 2560), (64, 4112)])
def test_rows(nv, orc, M, K):
    x = W.small_matrix(M * 3 + K, M, K, dist="student_t3", outlier_cols=min(3, K // 16))
    r = orc.quantize(x)
    got = _run(nv, r["q"], r["sf_swz"], r["s"], 1, M, K)
    want = orc.dequantize_bf16(r["q"], r["sf"], r["s"])
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} differ, first {bad[:5].tolist()}"


@pytest.mark.parametrize("M,K", [(96, 256), (400, 2048)])
def test_column_copy_single_scale(nv, orc, M, K):
    x = W.small_matrix(M + K, M, K, outlier_cols=2, outlier_scale=30)
    r = orc.quantize(x, column_copy=True)
    got = _run(nv, r["q_col"], r["sf_col_swz"], r["s_col"], 0, K, M)
    want = orc.dequantize_bf16(r["q_col"], r["sf_col"], r["s_col"], s_per_row=False)
    assert np.array_equal(got, want)


def test_padded_pitch_leaves_the_gap(nv, orc):
    x = W.small_matrix(5, 130, 512)
    r = orc.quantize(x)
    got = _run(nv, r["q"], r["sf_swz"], r["s"], 1, 130, 512, ld=520)
    assert np.array_equal(got[:, :512], orc.dequantize_bf16(r["q"], r["sf"], r["s"]))
    assert np.all(got[:, 512:] == np.uint16(0xFFFF))


def test_config2_activation_full(nv, orc):
    wl = W.config2()
    r = orc.quantize(wl.x)
    got = _run(nv, r["q"], r["sf_swz"], r["s"], 1, wl.x.shape[0], wl.x.shape[1])
    assert np.array_equal(got, orc.dequantize_bf16(r["q"], r["sf"], r["s"]))


def test_gpu_quantize_then_dequantize(nv, orc):
    """Through the binding: dequantize(quantize(x)) on the GPU equals the oracle's
    dequantization of the oracle's quantization of the same x."""
    x = W.small_matrix(77, 256, 1024, dist="lognormal_rows")
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    y = nv.dequantize(nv.quantize(xd))
    r = orc.quantize(x)
    assert np.array_equal(host(y), orc.dequantize_bf16(r["q"], r["sf"], r["s"]))


def test_empty_and_errors(nv):
    q = torch.zeros((4, 8), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(512, dtype=torch.uint8, device="cuda")
    s = torch.zeros(4, dtype=torch.float32, device="cuda")
    y = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_dequantize(q, sf, s, 1, 0, 16, y, 16)          # rows == 0: no-op
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_dequantize(q, sf, s, 1, 4, 24, y, 24)      # cols % 16 != 0
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_dequantize(q, sf, s, 1, 4, 16, y, 12)      # ld_y < cols
