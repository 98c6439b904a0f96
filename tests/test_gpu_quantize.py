"""GPU parity of the per-token quantizer against the CPU oracle: packed codes,
swizzled block scales and FP32 outer scales must be bit-identical.

Cases: small shapes spanning several row tiles with ragged tails (rows not a
multiple of 128, blocks per row not a multiple of 4, rows longer than the
register-resident path), the pages' four bit-exact test classes (random,
boundary, zeros, maxes: "Towards Blackwell-Native 8-bit and 4-bit RL",
"Bit-exact quantizer contract"), gather indices with padding, per-tensor mode,
the column-wise copy, and the five workloads at full size.
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import assert_quant_equal, host, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(1, 16), (7, 48), (130, 256), (257, 512), (300, 2560), (64, 4096), (33, 4112),
          (200, 768), (129, 2064)]


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("dist", ["normal", "student_t3", "lognormal_rows"])
def test_small_shapes(nv, orc, M, K, dist):
    x = W.small_matrix(M * 7 + K, M, K, dist=dist, outlier_cols=min(3, K // 16))
    got = nv.quantize(to_dev(x))
    assert_quant_equal(got, orc.quantize(x), what=f"{M}x{K} {dist}")


@pytest.mark.parametrize("kind", ["random", "boundary", "zeros", "maxes"])
@pytest.mark.parametrize("M,K", [(128, 256), (37, 1024), (300, 64)])
def test_init_data_classes(nv, orc, kind, M, K):
    x = W.init_data_class(kind, 5, M, K)
    got = nv.quantize(to_dev(x))
    assert_quant_equal(got, orc.quantize(x), what=f"{kind} {M}x{K}")


@pytest.mark.parametrize("M,K", [(508, 256), (508, 768), (254, 2048), (64, 8192)])
def test_rows_across_the_exponent_range(nv, orc, M, K):
    """Row scales from bf16 subnormals up to the bf16 maximum, every biased
    exponent at the top of some row, elements up to 40 binades below it: rows
    whose outer scale lies outside [2^-90, 2^90] take the IEEE form of the
    scale arithmetic, the others the FMA form; both give the oracle's bytes."""
    rng = np.random.Generator(np.random.PCG64(M * 31 + K))
    top = np.resize(np.arange(1, 255, dtype=np.int64), M) if M >= 254 else np.linspace(1, 254, M).astype(np.int64)
    e = np.clip(top[:, None] - rng.integers(0, 41, size=(M, K)), 0, 254)
    e[np.arange(M), rng.integers(0, K, size=M)] = top          # the row's top exponent is present
    mant = rng.integers(0, 128, size=(M, K))
    sign = rng.integers(0, 2, size=(M, K)) << 15
    x = (sign | (e << 7) | mant).astype(np.uint16)
    got = nv.quantize(to_dev(x))
    assert_quant_equal(got, orc.quantize(x), what=f"exponent range {M}x{K}")


def test_scale_recipe_fma_form_matches_ieee(nv):
    """The FMA form of the block-scale quotient and reciprocal against the IEEE
    intrinsics, on the GPU, over every (row amax, block amax <= row amax) pair of
    bf16 values; the number of pairs compared is the count of rows in the FMA
    range, computed here with numpy's IEEE binary32 division."""
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    bad = torch.zeros(17, dtype=torch.int32, device="cuda")
    nv.nvfp4_debug_scale_recipe_check(cnt, bad)
    torch.cuda.synchronize()
    c = cnt.cpu().numpy()
    b = bad.cpu().numpy().view(np.uint32)
    bits = np.arange(0x7F80, dtype=np.uint32)
    S = (bits << np.uint32(16)).view(np.float32) / np.float32(2688.0)
    fast = (S >= np.float32(2.0 ** -90)) & (S <= np.float32(2.0 ** 90))
    assert int(c[0]) == int(np.sum(bits[fast].astype(np.int64) + 1))
    pairs = [(hex(b[1 + 2 * k]), hex(b[2 + 2 * k])) for k in range(min(int(b[0]), 8))]
    assert int(c[1]) == 0, f"{int(c[1])} pairs differ, first {pairs}"


@pytest.mark.parametrize("M,K", [(96, 256), (160, 768), (400, 2048), (48, 4112)])
def test_per_tensor_and_column_copy(nv, orc, M, K):
    x = W.small_matrix(M + 3 * K, M, K, dist="student_t3", outlier_cols=4, outlier_scale=50)
    for mode in ("per_token", "per_tensor"):
        got = nv.quantize(to_dev(x), mode=mode, column_copy=True)
        ref = orc.quantize(x, mode=mode, column_copy=True)
        assert_quant_equal(got, ref, what=f"{mode} rows")
        assert_quant_equal(got, ref, what=f"{mode} columns", col=True)


def test_gather_with_padding_rows(nv, orc):
    x = W.small_matrix(9, 300, 512)
    rng = np.random.default_rng(0)
    g = rng.integers(-1, 300, size=1008).astype(np.int32)
    g[:5] = -1
    got = nv.quantize(to_dev(x), gather=torch.from_numpy(g).cuda(), column_copy=True)
    ref = orc.quantize(x, gather=g, column_copy=True)
    assert_quant_equal(got, ref, what="gather")
    assert_quant_equal(got, ref, what="gather columns", col=True)


def test_empty_and_all_padding(nv, orc):
    x = W.small_matrix(10, 4, 64)
    got = nv.quantize(to_dev(x), rows_out=0)
    assert got["q"].numel() == 0
    g = torch.full((16,), -1, dtype=torch.int32, device="cuda")
    got = nv.quantize(to_dev(x), gather=g, column_copy=True)
    assert not host(got["q"]).any() and not host(got["sf"]).any()
    assert not host(got["s"]).any() and host(got["s_col"])[0] == 0


def test_batch_invariance_on_gpu(nv):
    """Each token quantized alone on the GPU equals the same token in the batch."""
    x = W.small_matrix(11, 512, 2048, dist="student_t3", outlier_cols=8, outlier_scale=50)
    xd = to_dev(x)
    full = nv.quantize(xd)
    for r in (0, 1, 127, 128, 300, 511):
        alone = nv.quantize(xd[r:r + 1])
        assert torch.equal(alone["q"][0], full["q"][r])
        assert alone["s"][0].item() == full["s"][r].item()
    # per-tensor scales do depend on the batch
    pt_full = nv.quantize(xd, mode="per_tensor")
    pt_alone = nv.quantize(xd[300:301], mode="per_tensor")
    assert not torch.equal(pt_alone["q"][0], pt_full["q"][300])


def _full_config(nv, orc, x, what, column_copy=False, modes=("per_token",)):
    xd = to_dev(x)
    for mode in modes:
        got = nv.quantize(xd, mode=mode, column_copy=column_copy)
        ref = orc.quantize(x, mode=mode, column_copy=column_copy)
        assert_quant_equal(got, ref, what=f"{what} {mode}")
        if column_copy:
            assert_quant_equal(got, ref, what=f"{what} {mode} columns", col=True)
    del xd


def test_config1_full(nv, orc):
    wl = W.config1()
    _full_config(nv, orc, wl.x, "config1 X")
    _full_config(nv, orc, wl.w, "config1 W")


def test_config2_full(nv, orc):
    wl = W.config2()
    _full_config(nv, orc, wl.x, "config2 X", column_copy=True)
    _full_config(nv, orc, wl.w, "config2 W")


def test_config4_full(nv, orc):
    wl = W.config4()
    _full_config(nv, orc, wl.x, "config4 X", modes=("per_token", "per_tensor"))
    _full_config(nv, orc, wl.w, "config4 W")


def test_config5_full(nv, orc):
    wl = W.config5(moe=False)
    _full_config(nv, orc, wl.x, "config5 X")
    _full_config(nv, orc, wl.w, "config5 W")
