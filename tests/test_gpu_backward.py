"""GPU parity of the NVFP4 backward GEMMs (nvfp4_gemm_ex with column-wise
copies, one outer scale per operand copy):

  dgrad  dX = dY W      A = dY (rows, per-token scales), B = W's column-wise copy
  wgrad  dW = dY^T X    A = dY's column-wise copy, B = X's column-wise copy

against the oracle's exact product of the oracle's own quantizations (the
column copies' single scale broadcast to every row).  Tolerance as the forward
GEMM (tests/_gpu_util.check_gemm).
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import bf16_to_f64, check_gemm, to_dev

pytestmark = pytest.mark.gpu


def _col_operand(r):
    rows = r["q_col"].shape[0]
    return dict(q=r["q_col"], sf=r["sf_col"], s=np.full(rows, r["s_col"][0], np.float32))


def _inputs(M, N, K, seed):
    x = W.small_matrix(seed, M, K, dist="student_t3", outlier_cols=2, outlier_scale=20)
    w = W.small_matrix(seed + 1, N, K, std=0.02)
    dy = W.small_matrix(seed + 2, M, N, std=1e-3)
    return x, w, dy


@pytest.mark.parametrize("M,N,K", [(256, 512, 320), (384, 128, 1024), (1024, 640, 256)])
def test_dgrad_and_wgrad_small(nv, orc, M, N, K):
    x, w, dy = _inputs(M, N, K, M + N + K)
    qx = nv.quantize(to_dev(x), column_copy=True)
    qw = nv.quantize(to_dev(w), column_copy=True)
    qdy = nv.quantize(to_dev(dy), column_copy=True)
    dx = nv.gemm_dgrad(qdy, qw)
    dw = nv.gemm_wgrad(qdy, qx)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    rx, rw, rdy = (orc.quantize(t, column_copy=True) for t in (x, w, dy))
    ref, absr = orc.gemm_exact(rdy, _col_operand(rw), with_abs=True)       # [M, K]
    check_gemm(bf16_to_f64(dx), ref, absr, N, f"dgrad {M}x{N}x{K}")
    ref, absr = orc.gemm_exact(_col_operand(rdy), _col_operand(rx), with_abs=True)   # [N, K]
    check_gemm(bf16_to_f64(dw), ref, absr, M, f"wgrad {M}x{N}x{K}")


def test_qwen3_4b_up_projection_backward_sampled(nv, orc):
    wl = W.config2()
    M, K = wl.x.shape
    N = wl.w.shape[0]
    dy = W.small_matrix(77, M, N, std=1e-3)
    qx = nv.quantize(to_dev(wl.x), column_copy=True)
    qw = nv.quantize(to_dev(wl.w), column_copy=True)
    qdy = nv.quantize(to_dev(dy), column_copy=True)
    dx = bf16_to_f64(nv.gemm_dgrad(qdy, qw))
    dw = bf16_to_f64(nv.gemm_wgrad(qdy, qx))
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    rng = np.random.default_rng(5)
    rdy = orc.quantize(dy, column_copy=True)
    rw = orc.quantize(wl.w, column_copy=True)
    rx = orc.quantize(wl.x, column_copy=True)
    mi, ki = rng.integers(0, M, 3000), rng.integers(0, K, 3000)
    ref, absr = orc.gemm_exact_sampled(rdy, _col_operand(rw), mi, ki)
    check_gemm(dx[mi, ki], ref, absr, N, "dgrad config 2")
    ni, ki = rng.integers(0, N, 3000), rng.integers(0, K, 3000)
    ref, absr = orc.gemm_exact_sampled(_col_operand(rdy), _col_operand(rx), ni, ki)
    check_gemm(dw[ni, ki], ref, absr, M, "wgrad config 2")


def test_per_row_flags_match_the_forward_gemm(nv):
    x, w, _ = _inputs(200, 256, 512, 9)
    a, b = nv.quantize(to_dev(x)), nv.quantize(to_dev(w))
    assert torch.equal(nv.gemm_ex(a, b), nv.gemm(a, b))
