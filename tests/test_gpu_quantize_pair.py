"""GPU parity of nvfp4_quantize_per_token_pair: an activation (with and without
its column-wise copy) and a weight with the same K quantized in one launch must
give, for each tensor, exactly the oracle's bytes of that tensor quantized alone.
Shapes span ragged row counts on both sides, an empty side, the Qwen3-4B
up-projection (K = 2560) and a K past the staged kernel's range (two launches).
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import assert_quant_equal, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Mx,Mw,K,col", [(144, 257, 512, True), (130, 129, 512, False), (96, 40, 2560, True), (4096, 9728, 2560, True),
                                         (33, 300, 1040, False), (64, 200, 4112, True), (0, 77, 256, False),
                                         (48, 0, 256, True)])
def test_pair_equals_each_alone(nv, orc, Mx, Mw, K, col):
    x = W.small_matrix(Mx + K, Mx, K, dist="student_t3", outlier_cols=min(3, K // 16), outlier_scale=40)
    w = W.small_matrix(Mw + 2 * K, Mw, K, std=0.02)
    ox, ow = nv.quantize_pair(to_dev(x), to_dev(w), column_copy=col)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    if Mx:
        rx = orc.quantize(x, column_copy=col)
        assert_quant_equal(ox, rx, what="x rows")
        if col:
            assert_quant_equal(ox, rx, what="x columns", col=True)
    if Mw:
        assert_quant_equal(ow, orc.quantize(w), what="w rows")


def test_pair_matches_single_calls_on_gpu(nv):
    wl = W.config2()
    x, w = to_dev(wl.x), to_dev(wl.w)
    ox, ow = nv.quantize_pair(x, w, column_copy=True)
    sx, sw = nv.quantize(x, column_copy=True), nv.quantize(w)
    for k in ("q", "sf", "s", "q_col", "sf_col", "s_col"):
        assert torch.equal(ox[k], sx[k]), k
    for k in ("q", "sf", "s"):
        assert torch.equal(ow[k], sw[k]), k
