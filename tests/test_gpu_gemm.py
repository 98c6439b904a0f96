"""GPU parity of the dense W4A4 GEMM (tcgen05 block-scaled MMA) against the
oracle's exact integer GEMM on the same quantized operands.

Tolerance (the reading of "max relative error 2e-3 after bf16 rounding"):
normwise relative error <= 2e-3, and every element within one bf16 ulp of the
exact value plus a 4*K*2^-24 FP32-summation allowance (tests/_gpu_util.py).

Besides quantizer-fed cases, two hand-built operand sets pin the MMA operand
layout independently of the quantizer: codes in {0, +1, -1} with unit scales
(an integer matmul, exact in bf16), and unit codes with random block scales
(the sum of per-block scale products, which pins the swizzled scale layout).
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import bf16_to_f64, check_gemm, host, to_dev

pytestmark = pytest.mark.gpu


def _run(nv, orc, x, w, what, sample=None):
    a, b = nv.quantize(to_dev(x)), nv.quantize(to_dev(w))
    y = nv.gemm(a, b)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    # the oracle quantizes the same bf16 inputs itself (never the GPU's bytes)
    ra, rb = orc.quantize(x), orc.quantize(w)
    K = a["cols"]
    if sample is None:
        yref, absy = orc.gemm_exact(ra, rb, with_abs=True)
        return check_gemm(bf16_to_f64(y), yref, absy, K, what)
    mi, ni = sample
    yref, absy = orc.gemm_exact_sampled(ra, rb, mi, ni)
    yg = bf16_to_f64(y)[mi, ni]
    return check_gemm(yg, yref, absy, K, what)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (1, 16, 64), (130, 272, 320), (257, 512, 1024),
                                   (384, 768, 2048), (96, 256, 4096), (200, 400, 192)])
def test_small_shapes(nv, orc, M, N, K):
    x = W.small_matrix(M + N + K, M, K, outlier_cols=2)
    w = W.small_matrix(M * N + K, N, K, std=0.02)
    _run(nv, orc, x, w, f"{M}x{N}x{K}")


def _pack(codes):
    codes = codes.astype(np.uint8)
    return np.ascontiguousarray(codes[:, 0::2] | (codes[:, 1::2] << 4))


def _swizzle(sf_rm):
    """Documented 128 x 4 scale tile layout, written out here so that these
    hand-built operands depend on neither the oracle nor the GPU quantizer."""
    rows, kb = sf_rm.shape
    kb4 = -(-kb // 4) * 4
    out = np.zeros((-(-rows // 128) * 128) * kb4, np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(kb), indexing="ij")
    off = ((r // 128) * (kb4 // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
    out[off.ravel()] = sf_rm.ravel()
    return out


def _operand(nv, orc, codes, sf_rm, s):
    rows, K = codes.shape
    q = torch.from_numpy(_pack(codes)).cuda()
    sf = torch.from_numpy(_swizzle(sf_rm)).cuda()
    return dict(rows=rows, cols=K, q=q, sf=sf, s=torch.from_numpy(s.astype(np.float32)).cuda())


def test_integer_operands_exact(nv, orc):
    rng = np.random.default_rng(1)
    M, N, K = 256, 512, 128
    ia = rng.choice([0, 1, -1], size=(M, K))
    ib = rng.choice([0, 1, -1], size=(N, K))
    enc = {0: 0, 1: 2, -1: 10}
    ca = np.vectorize(enc.get)(ia)
    cb = np.vectorize(enc.get)(ib)
    ones_a = np.full((M, K // 16), 0x38, np.uint8)
    ones_b = np.full((N, K // 16), 0x38, np.uint8)
    a = _operand(nv, orc, ca, ones_a, np.ones(M))
    b = _operand(nv, orc, cb, ones_b, np.ones(N))
    y = bf16_to_f64(nv.gemm(a, b))
    assert np.array_equal(y, (ia @ ib.T).astype(np.float64))


def test_block_scale_placement(nv, orc):
    """Unit codes, random power-of-two block scales: Y = 16 * sum_b sa_b * sb_b."""
    rng = np.random.default_rng(2)
    M, N, K = 256, 512, 512
    kb = K // 16
    ea = rng.integers(-3, 4, size=(M, kb))
    eb = rng.integers(-3, 4, size=(N, kb))
    sfa = (0x38 + 8 * ea).astype(np.uint8)      # E4M3 code of 2^e
    sfb = (0x38 + 8 * eb).astype(np.uint8)
    a = _operand(nv, orc, np.full((M, K), 2), sfa, np.ones(M))
    b = _operand(nv, orc, np.full((N, K), 2), sfb, np.ones(N))
    y = bf16_to_f64(nv.gemm(a, b))
    ref = 16.0 * (2.0 ** ea) @ (2.0 ** eb).T
    assert np.all(np.abs(y - ref) <= ref * 2.0 ** -8)


def test_outer_scales_in_epilogue(nv, orc):
    rng = np.random.default_rng(3)
    M, N, K = 128, 256, 64
    a = _operand(nv, orc, np.full((M, K), 2), np.full((M, 4), 0x38, np.uint8),
                 2.0 ** rng.integers(-10, 10, M))
    b = _operand(nv, orc, np.full((N, K), 2), np.full((N, 4), 0x38, np.uint8),
                 2.0 ** rng.integers(-10, 10, N))
    y = bf16_to_f64(nv.gemm(a, b))
    ref = 64.0 * np.outer(host(a["s"]).astype(np.float64), host(b["s"]).astype(np.float64))
    assert np.array_equal(y, ref)


def test_config1_full(nv, orc):
    wl = W.config1()
    _run(nv, orc, wl.x, wl.w, "config1")


def _sample(rng, M, N, n=6000):
    mi = np.concatenate([rng.integers(0, M, n), np.full(256, M - 1), np.arange(256) % M])
    ni = np.concatenate([rng.integers(0, N, n), np.arange(256) % N, np.full(256, N - 1)])
    return mi, ni


def test_config2_sampled(nv, orc):
    wl = W.config2()
    _run(nv, orc, wl.x, wl.w, "config2", sample=_sample(np.random.default_rng(4), 4096, 9728))


def test_config4_sampled(nv, orc):
    wl = W.config4()
    _run(nv, orc, wl.x, wl.w, "config4", sample=_sample(np.random.default_rng(5), 16384, 4096))


def test_config5_sampled(nv, orc):
    wl = W.config5(moe=False)
    _run(nv, orc, wl.x, wl.w, "config5", sample=_sample(np.random.default_rng(6), 65536, 6144))


def test_gemm_abort_path_records_timeout_and_context_stays_usable(nv):
    """With the GEMM pipeline wait limit set to 1 ns (every wait that is not
    complete at its first attempt gives up; the limit is enforced at the
    resolution of the GPU's global timer), a dense and a grouped GEMM each
    record NVFP4_ERR_TIMEOUT and return: every role of both CTAs leaves its
    loop, copies and MMAs in flight complete, TMEM is freed.  With the default
    limit restored, the same GEMMs in the same context give the same bytes as
    before into freshly poisoned outputs."""
    import time
    x = torch.randn(4096, 2560, device="cuda").to(torch.bfloat16)
    w = (torch.randn(9728, 2560, device="cuda") * 0.02).to(torch.bfloat16)
    a, b = nv.quantize(x), nv.quantize(w)
    T, H, N, E, k = 2048, 1024, 512, 16, 4
    ids = torch.from_numpy(W.route_topk(np.random.default_rng(5), T, E, k)).cuda()
    perm = nv.moe_permute(ids, E, row_align=256)
    ga = nv.quantize(torch.randn(T, H, device="cuda").to(torch.bfloat16), gather=perm["gather"])
    gw = nv.quantize_experts((torch.randn(E, N, H, device="cuda") * 0.02).to(torch.bfloat16))
    y = torch.empty(4096, 9728, dtype=torch.bfloat16, device="cuda")
    yg = torch.empty(ga["rows"], N, dtype=torch.bfloat16, device="cuda")

    def run():
        y.view(torch.int16).fill_(0x7FC1)          # NaN: nothing left over from an earlier call
        yg.view(torch.int16).fill_(0x7FC1)
        nv.gemm(a, b, out=y)
        nv.grouped_gemm(ga, perm["offsets"], E, gw["q"], gw["sf"], gw["s"], N, H, out=yg)
        torch.cuda.synchronize()
    run()
    assert nv.nvfp4_get_device_status() == 0
    used = int(perm["offsets"][E].item())
    ref, refg = y.clone(), yg[:used].clone()
    statuses = []
    try:
        nv.nvfp4_debug_set_gemm_wait_limit(1)
        for fn in (lambda: nv.gemm(a, b, out=y),
                   lambda: nv.grouped_gemm(ga, perm["offsets"], E, gw["q"], gw["sf"], gw["s"], N, H, out=yg)):
            t0 = time.time()
            fn()
            torch.cuda.synchronize()
            statuses.append((nv.nvfp4_get_device_status(), time.time() - t0 < 5.0))
    finally:
        nv.nvfp4_debug_set_gemm_wait_limit(0)
    assert statuses == [(6, True), (6, True)], statuses    # NVFP4_ERR_TIMEOUT, returned promptly
    run()
    assert nv.nvfp4_get_device_status() == 0
    assert torch.equal(y, ref) and torch.equal(yg[:used], refg)
