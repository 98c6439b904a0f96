"""GPU parity of nvfp4_moe_combine (unpermute + weighted combine) against the
oracle, bit-exact: binary32 reduction in slot order on both sides.

Cases: the Qwen3-30B-A3B expert step at 4096 tokens (top-8, hidden 2048, the
permutation of its seeded routing), runtime top-k values (1 and 3), a hidden
size that is not a multiple of 64, a padded output pitch, rows outside the
layout (contribute nothing, device status DEVICE_INPUT) and empty input.
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import host

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bf16(bits):
    return _dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _case(nv, orc, y2, dst, w, ld_out=None):
    T, K = w.shape
    H = y2.shape[1]
    ld_out = H if ld_out is None else ld_out
    out = torch.full((T, ld_out), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    nv.nvfp4_moe_combine(_bf16(y2), y2.shape[0], H, _dev(dst.astype(np.int32)), _dev(w), T, K, H, out, ld_out)
    torch.cuda.synchronize()
    return host(out)


def test_qwen3_moe_step_full(nv, orc):
    wl = W.config3(weights=False)
    m = wl.moe
    perm = orc.moe_permute(m.topk_ids, m.experts, align=128)
    rng = np.random.default_rng(11)
    y2 = W.to_bf16_bits(rng.standard_normal((perm["capacity"], m.hidden)).astype(np.float32))
    w = W.topk_weights(2, m.tokens, m.topk)
    got = _case(nv, orc, y2, perm["dst"], w)
    assert nv.nvfp4_get_device_status() == 0
    want = orc.moe_combine(y2, perm["dst"], w)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} differ, first {bad[:5].tolist()}"


@pytest.mark.parametrize("T,K,H", [(37, 1, 64), (100, 3, 24), (513, 8, 2056), (77, 8, 272), (5, 8, 16), (20000, 8, 512)])
def test_small_shapes(nv, orc, T, K, H):
    """Top-k weighted combine on random rows; (20000, 8, 512) has enough 8-column
    chunk pairs for the two-chunk kernel on a 152-SM GPU."""
    rng = np.random.default_rng(T * K + H)
    R = 3 * T + 7
    y2 = W.to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    dst = rng.integers(0, R, size=(T, K)).astype(np.int32)
    w = W.topk_weights(T, T, K)
    got = _case(nv, orc, y2, dst, w, ld_out=H + 8)
    assert nv.nvfp4_get_device_status() == 0
    assert np.array_equal(got[:, :H], orc.moe_combine(y2, dst, w))
    assert np.all(got[:, H:] == np.uint16(0xFFFF))


def test_rows_outside_the_layout(nv, orc):
    rng = np.random.default_rng(12)
    y2 = W.to_bf16_bits(rng.standard_normal((50, 32)).astype(np.float32))
    dst = rng.integers(0, 50, size=(20, 4)).astype(np.int32)
    dst[3, 1] = -1
    dst[7, 2] = 50
    w = W.topk_weights(3, 20, 4)
    got = _case(nv, orc, y2, dst, w)
    assert nv.nvfp4_get_device_status() == 7          # NVFP4_ERR_DEVICE_INPUT
    assert nv.nvfp4_get_device_status() == 0          # reading it clears it
    assert np.array_equal(got, orc.moe_combine(y2, dst, w))


def test_empty_and_errors(nv):
    y2 = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    dst = torch.zeros(8, dtype=torch.int32, device="cuda")
    w = torch.zeros((4, 2), dtype=torch.float32, device="cuda")
    out = torch.zeros((4, 16), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_moe_combine(y2, 4, 16, dst, w, 0, 2, 16, out, 16)        # no tokens: no-op
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_moe_combine(y2, 4, 16, dst, w, 4, 2, 12, out, 16)    # hidden % 8 != 0
    with pytest.raises(nv.NVFP4Error):
        nv.nvfp4_moe_combine(y2, 4, 16, dst, w, 4, 33, 16, out, 16)   # topk > 32
