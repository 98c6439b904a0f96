"""GPU parity of the MoE path: routing permute (bit-exact), gather-quantize into
the padded per-expert layout (bit-exact), fused SwiGLU + quantize, and the
grouped W4A4 GEMM (tolerance of the dense GEMM), each on seeded inputs that
the oracle also receives.  Workload: Qwen3-30B-A3B-shaped experts (hidden 2048,
expert FFN 768, 128 experts, top-8), as on "Towards Blackwell-Native 8-bit and
4-bit RL" ("Experimental setup": Qwen3-30B-A3B; routed experts fc1 / fc2 are
the NVFP4 layers of the recipe).
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import assert_quant_equal, bf16_to_f64, bf16_ulp, check_gemm, host, to_dev

pytestmark = pytest.mark.gpu


def _ids(seed, T, E, k):
    return W.route_topk(np.random.default_rng(seed), T, E, k)


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (37, 8, 2), (300, 16, 4), (40, 64, 2),
                                   (4096, 128, 8), (65536, 128, 8),
                                   # 64 and 65 chunks of 1,024 ids: the two sides of the
                                   # switch from the one-block scan to one block per expert
                                   (8192, 128, 8), (8320, 128, 8), (8320, 1000, 8)])
def test_permute_bit_exact(nv, orc, T, E, k):
    ids = _ids(T + E, T, E, k)
    got = nv.moe_permute(torch.from_numpy(ids).cuda(), E)
    ref = orc.moe_permute(ids, E, 128, capacity=got["capacity"])
    assert np.array_equal(host(got["offsets"]), ref["offsets"])
    assert np.array_equal(host(got["gather"]), ref["gather"])
    assert np.array_equal(host(got["dst"]), ref["dst"])
    assert nv.nvfp4_get_device_status() == 0


def test_permute_reports_bad_ids(nv):
    ids = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    got = nv.moe_permute(ids, 4)
    assert nv.nvfp4_get_device_status() == 7          # NVFP4_ERR_DEVICE_INPUT
    dst = host(got["dst"])
    assert dst[1, 1] == -1 and (dst[0] >= 0).all()


def test_gather_quantize_bit_exact(nv, orc):
    T, H, E, k = 300, 512, 16, 4
    x = W.small_matrix(21, T, H)
    ids = _ids(22, T, E, k)
    perm = nv.moe_permute(torch.from_numpy(ids).cuda(), E)
    rperm = orc.moe_permute(ids, E, 128, capacity=perm["capacity"])
    got = nv.quantize(to_dev(x), gather=perm["gather"])
    ref = orc.quantize(x, gather=rperm["gather"])
    assert_quant_equal(got, ref, what="gather-quantize")


@pytest.mark.parametrize("T,H,E,k,align", [(300, 512, 16, 4, 128), (100, 272, 8, 2, 256),
                                           (4096, 2048, 128, 8, 256)])
def test_gather_quantized_bit_exact(nv, orc, T, H, E, k, align):
    """Quantize the tokens once, then scatter the quantized rows to the routed
    layout: equal, bit for bit, to quantizing the gathered rows."""
    x = W.small_matrix(23 + T, T, H, dist="lognormal_rows")
    ids = _ids(24 + T, T, E, k)
    perm = nv.moe_permute(torch.from_numpy(ids).cuda(), E, row_align=align)
    rperm = orc.moe_permute(ids, E, align, capacity=perm["capacity"])
    got = nv.moe_gather_quantized(nv.quantize(to_dev(x)), perm["gather"], perm["offsets"])
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    ref = orc.quantize(x, gather=rperm["gather"])
    assert_quant_equal(got, ref, what="gather of quantized rows")


@pytest.mark.parametrize("T,H,E,k,align", [(300, 512, 16, 4, 128), (4096, 2048, 128, 8, 256)])
@pytest.mark.parametrize("order", ["none", "foreign", "unaligned", "decreasing", "too_many"])
def test_gather_quantized_tile_order(nv, orc, T, H, E, k, align, order):
    """The expert offsets only order the tiles: with none, with offsets of
    another layout (non-decreasing, starting past 0, ending short of the rows),
    with unaligned or decreasing ones, or more experts than the order handles,
    every byte is the same as the oracle's gather-quantize."""
    x = W.small_matrix(25 + T, T, H, dist="lognormal_rows")
    ids = _ids(26 + T, T, E, k)
    perm = nv.moe_permute(torch.from_numpy(ids).cuda(), E, row_align=align)
    rows = perm["capacity"]
    rng = np.random.default_rng(27 + T)
    if order == "none":
        offs = None
    elif order == "foreign":
        o = np.sort(rng.integers(128, max(rows - 200, 129), size=E + 1)).astype(np.int32)
        offs = torch.from_numpy(o).cuda()
    elif order == "unaligned":
        o = np.sort(rng.integers(0, rows + 1000, size=E + 1)).astype(np.int32)
        o[0] = 3
        offs = torch.from_numpy(o).cuda()
    elif order == "decreasing":
        o = host(perm["offsets"]).copy()
        o[E // 2] = o[E // 2 + 1] + 1
        offs = torch.from_numpy(o).cuda()
    else:
        offs = torch.arange(0, 300 * 128, 128, dtype=torch.int32, device="cuda")   # 299 experts
    got = nv.moe_gather_quantized(nv.quantize(to_dev(x)), perm["gather"], offs)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    rperm = orc.moe_permute(ids, E, align, capacity=rows)
    ref = orc.quantize(x, gather=rperm["gather"])
    assert_quant_equal(got, ref, what=f"gather of quantized rows ({order} order)")


def test_gather_quantized_bad_index(nv):
    q = nv.quantize(torch.randn(8, 64, device="cuda").to(torch.bfloat16))
    g = torch.tensor([0, 7, 8, -1], dtype=torch.int32, device="cuda")
    out = nv.moe_gather_quantized(q, g)
    assert nv.nvfp4_get_device_status() == 7          # NVFP4_ERR_DEVICE_INPUT
    assert not out["q"][2:].any() and not out["s"][2:].any()
    assert torch.equal(out["q"][1], q["q"][7]) and out["s"][1] == q["s"][7]


@pytest.mark.parametrize("R,F", [(300, 768), (77, 768), (200, 640), (129, 64), (64, 2048)])
def test_swiglu_quantize(nv, orc, R, F):
    rng = np.random.default_rng(R + F)
    y1 = W.to_bf16_bits((rng.standard_normal((R, 2 * F)) * 2).astype(np.float32))
    got = nv.swiglu_quantize(to_dev(y1), F, want_h=True)
    h_ref = orc.swiglu(y1, F)
    hg = bf16_to_f64(got["h"])
    hr = W.bf16_bits_to_float(h_ref).astype(np.float64)
    assert np.all(np.abs(hg - hr) <= bf16_ulp(hr)), "h differs by more than one bf16 ulp"
    # rows whose h agrees exactly quantize bit-exactly; the fused quantize is
    # the row quantizer's own code, checked against the GPU row quantizer too
    ref = orc.quantize(h_ref)
    hb = host(got["h"]).view(np.uint16)
    same = np.all(hb == h_ref, axis=1)
    # measured: about 1e-5 of h values one ulp from the correctly rounded one
    # (the binary32 silu's error straddling a bf16 rounding midpoint)
    assert np.mean(hb != h_ref) < 1e-4 and same.mean() > 0.9
    assert_quant_equal(got, ref, rows=np.nonzero(same)[0], what="swiglu rows")
    again = nv.quantize(got["h"])
    assert torch.equal(again["q"], got["q"]) and torch.equal(again["sf"], got["sf"])
    assert torch.equal(again["s"], got["s"])


def test_swiglu_gate_tails(nv, orc):
    """h within one bf16 ulp of the exact bf16(silu(g) u) across the gate's
    range, including large negative gates where exp(-g) would overflow and
    silu(g) is far below 1 (scaled up by large up-projection values)."""
    F = 256
    g = np.concatenate([np.linspace(-90.0, -20.0, 96), np.linspace(-20.0, 20.0, 128),
                        np.linspace(20.0, 90.0, 32)]).astype(np.float32)
    us = np.array([1.0, -1.0, 3.5, -300.0, 1.0e4, -1.0e4, 2.0 ** -60, 6.0e30], np.float32)
    y1 = np.zeros((us.size, 2 * F), np.float32)
    y1[:, :F] = g
    y1[:, F:] = us[:, None]
    bits = W.to_bf16_bits(y1)
    got = nv.swiglu_quantize(to_dev(bits), F, want_h=True)
    hg = bf16_to_f64(got["h"])
    hr = W.bf16_bits_to_float(orc.swiglu(bits, F)).astype(np.float64)
    bad = np.abs(hg - hr) > bf16_ulp(hr)
    assert not bad.any(), f"{bad.sum()} values off by more than one bf16 ulp, e.g. g={np.nonzero(bad)}"


def test_swiglu_row_count(nv):
    R, F = 256, 256
    y1 = torch.randn(R, 2 * F, device="cuda").to(torch.bfloat16)
    rc = torch.tensor([200], dtype=torch.int32, device="cuda")
    got = nv.swiglu_quantize(y1, F, row_count=rc, want_h=True)
    assert not got["h"][200:].any() and not got["q"][200:].any() and not got["s"][200:].any()
    assert got["s"][:200].gt(0).all()


def _grouped_case(nv, orc, T, H, N, E, k, seed, sample=None, align=128):
    """Grouped GEMM over a seeded routing; every expert is checked, in full or
    (sample) on that many random outputs plus its first and last valid rows and
    columns.  Only the used rows of the output are read back: rows past
    offsets[E] are not written."""
    x = W.small_matrix(seed, T, H)
    w = W.small_matrix(seed + 1, E * N, H, std=0.02).reshape(E, N, H)
    ids = _ids(seed + 2, T, E, k)
    perm = nv.moe_permute(torch.from_numpy(ids).cuda(), E, row_align=align)
    a = nv.quantize(to_dev(x), gather=perm["gather"])
    wq = nv.quantize_experts(to_dev(w.reshape(E * N, H)).reshape(E, N, H))
    y = nv.grouped_gemm(a, perm["offsets"], E, wq["q"], wq["sf"], wq["s"], N, H)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    rperm = orc.moe_permute(ids, E, align, capacity=perm["capacity"])
    assert np.array_equal(perm["offsets"].cpu().numpy(), rperm["offsets"])
    off, g = rperm["offsets"], rperm["gather"]
    used = int(off[E])
    yg = bf16_to_f64(y[:used])
    rx = orc.quantize(x)
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        pad = g[r0:r1] < 0
        if sample is None:
            ae = orc.rows_of(orc.quantize(x, gather=g[r0:r1]), 0, r1 - r0)
            yref, absy = orc.gemm_exact(ae, orc.quantize(w[e]), with_abs=True)
            check_gemm(yg[r0:r1], yref, absy, H, f"expert {e}")
        else:
            rng = np.random.default_rng(e)
            rows = np.nonzero(~pad)[0]
            mi = np.concatenate([rng.choice(rows, sample), rows[[0, -1, -1, 0]]])
            ni = np.concatenate([rng.integers(0, N, sample), [0, N - 1, 0, N - 1]])
            toks = g[r0 + mi]
            ar = dict(q=rx["q"][toks], sf=rx["sf"][toks], s=rx["s"][toks])
            idx = np.arange(mi.size)
            yref, absy = orc.gemm_exact_sampled(ar, orc.quantize(w[e][ni]), idx, idx)
            check_gemm(yg[r0 + mi, ni], yref, absy, H, f"expert {e}")
        assert not yg[r0:r1][pad].any()


@pytest.mark.parametrize("T,H,N,E,k", [(300, 256, 384, 16, 4), (40, 512, 256, 64, 2),
                                       (500, 768, 272, 8, 2)])
def test_grouped_gemm_small(nv, orc, T, H, N, E, k):
    _grouped_case(nv, orc, T, H, N, E, k, seed=T + N)


@pytest.mark.parametrize("T,H,N,E,k", [(300, 256, 384, 16, 4), (40, 512, 256, 64, 2)])
def test_grouped_gemm_256_aligned(nv, orc, T, H, N, E, k):
    """Expert segments padded to 256 rows: the kernel walks 256-row slots."""
    _grouped_case(nv, orc, T, H, N, E, k, seed=T + N + 7, align=256)


def test_grouped_fc1_config3_sampled_256_aligned(nv, orc):
    """fc1 at the full 4096-token, 128-expert size, 256-row layout: every expert."""
    _grouped_case(nv, orc, 4096, 2048, 1536, 128, 8, seed=33, sample=24, align=256)


def test_grouped_fc1_config3_sampled(nv, orc):
    """fc1 (gate+up, K=2048 -> N=1536) at the full size, 128-row layout: every expert."""
    _grouped_case(nv, orc, 4096, 2048, 1536, 128, 8, seed=31, sample=24)


def test_grouped_fc2_config3_sampled(nv, orc):
    """fc2 (down, K=768 -> N=2048) at the full size, on seeded expert inputs: every expert."""
    _grouped_case(nv, orc, 4096, 768, 2048, 128, 8, seed=41, sample=24)


def test_grouped_fc2_config3_sampled_256_aligned(nv, orc):
    _grouped_case(nv, orc, 4096, 768, 2048, 128, 8, seed=43, sample=24, align=256)


def _silu_h_bound(g, u, dg, du):
    """|h - silu(g) u| allowed when g and u are each off by dg, du, plus one bf16
    ulp of h and binary32 evaluation slack: silu'(g) = s (1 + g (1 - s)), s = sigma(g)."""
    s = 1.0 / (1.0 + np.exp(-np.clip(g, -700, 700)))
    h = g * s * u
    dsilu = np.abs(s * (1.0 + g * (1.0 - s)))
    return np.abs(u) * dsilu * dg + np.abs(g * s) * du + 2.0 * bf16_ulp(h) + 1e-6 * np.abs(h)


def _swiglu_case(nv, orc, T, H, F, E, k, seed, align, sample=None):
    """fc1 with the SwiGLU epilogue: (1) the same bits as the grouped GEMM
    followed by the SwiGLU kernel's h; rows past offsets[E] zero; (2) h within
    the GEMM tolerance, carried through silu(g) u, of the exact product."""
    x = W.small_matrix(seed, T, H)
    w = W.small_matrix(seed + 1, E * 2 * F, H, std=0.02).reshape(E, 2 * F, H)
    ids = _ids(seed + 2, T, E, k)
    perm = nv.moe_permute(torch.from_numpy(ids).cuda(), E, row_align=align)
    a = nv.quantize(to_dev(x), gather=perm["gather"])
    wq = nv.quantize_experts(to_dev(w.reshape(E * 2 * F, H)).reshape(E, 2 * F, H))
    y1 = nv.grouped_gemm(a, perm["offsets"], E, wq["q"], wq["sf"], wq["s"], 2 * F, H)
    ref = nv.swiglu_quantize(y1, F, row_count=perm["offsets"][E:], want_h=True)
    h = torch.full((a["rows"], F), 7, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    nv.grouped_gemm_swiglu(a, perm["offsets"], E, wq["q"], wq["sf"], wq["s"], F, H, out=h)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    used = int(perm["offsets"][E].item())
    assert torch.equal(h[:used].view(torch.int16), ref["h"][:used].view(torch.int16)), \
        "SwiGLU epilogue differs from the grouped GEMM + SwiGLU kernel"
    assert not h[used:].view(torch.int16).any(), "rows past the layout not zero"
    # against the oracle's exact products
    rperm = orc.moe_permute(ids, E, align, capacity=perm["capacity"])
    off, g = rperm["offsets"], rperm["gather"]
    rx = orc.quantize(x)
    hb = bf16_to_f64(h[:used])
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        rows = np.nonzero(g[r0:r1] >= 0)[0]
        rng = np.random.default_rng(100 + e)
        n = rows.size * F if sample is None else sample
        mi = rows[rng.integers(0, rows.size, n)] if sample else np.repeat(rows, F)
        ji = rng.integers(0, F, n) if sample else np.tile(np.arange(F), rows.size)
        toks = g[r0 + mi]
        ar = dict(q=rx["q"][toks], sf=rx["sf"][toks], s=rx["s"][toks])
        idx = np.arange(n)
        gq = orc.quantize(w[e][ji])
        uq = orc.quantize(w[e][F + ji])
        gr, ga = orc.gemm_exact_sampled(ar, gq, idx, idx)
        ur, ua = orc.gemm_exact_sampled(ar, uq, idx, idx)
        dg = bf16_ulp(gr) + 4.0 * H * 2.0 ** -24 * ga
        du = bf16_ulp(ur) + 4.0 * H * 2.0 ** -24 * ua
        s = 1.0 / (1.0 + np.exp(-np.clip(gr, -700, 700)))
        hx = gr * s * ur
        got = hb[r0 + mi, ji]
        bad = np.abs(got - hx) > _silu_h_bound(gr, ur, dg, du)
        assert not bad.any(), f"expert {e}: {bad.sum()} h values outside the carried GEMM tolerance"


@pytest.mark.parametrize("T,H,F,E,k,align", [(300, 256, 128, 16, 4, 128), (200, 512, 256, 8, 2, 256),
                                             (64, 192, 384, 4, 1, 128)])
def test_grouped_swiglu_small(nv, orc, T, H, F, E, k, align):
    _swiglu_case(nv, orc, T, H, F, E, k, seed=T + F, align=align)


def test_grouped_swiglu_config3(nv, orc):
    """fc1 (2048 -> 2 x 768) with the SwiGLU epilogue at 4096 tokens, 128
    experts, top-8, 256-row layout; every expert sampled."""
    _swiglu_case(nv, orc, 4096, 2048, 768, 128, 8, seed=61, align=256, sample=24)
