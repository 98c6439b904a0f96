"""GPU parity of the MoE half of the variable-length rollout workload: the
Qwen3-30B-A3B experts (hidden 2048, expert FFN 768, 128 experts, top-8) at
65,536 tokens, i.e. 524,288 routed rows in the 256-row aligned per-expert
layout the benchmark uses ("Towards Blackwell-Native 8-bit and 4-bit RL",
"Recipe 2: design of per-token NVFP4 RL": NVFP4 on the MoE experts).

Every stage gets seeded inputs that the oracle receives too (never the GPU's
output of the previous stage):
  permute           the workload's routing, bit-exact;
  quantize + gather the workload's tokens, quantized once and copied to the
                    layout, bit-exact against the oracle's quantization of the
                    tokens placed by the oracle's permutation;
  fc1 / fc2         the workload's expert weights, sampled outputs in EVERY
                    expert (first and last rows and columns included) at the
                    GEMM tolerance; pad rows must come out zero;
  SwiGLU + quantize a seeded full-size fc1 output, sampled rows: h within one
                    bf16 ulp, the quantized bytes bit-exact on rows whose h
                    agrees, rows past the layout zero;
  combine           a seeded full-size fc2 output, sampled tokens, bit-exact.
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W
from _gpu_util import bf16_ulp, check_gemm, host, to_dev

pytestmark = pytest.mark.gpu

ALIGN = 256
SAMPLES_PER_EXPERT = 24


@pytest.fixture(scope="module")
def rollout(nv, orc):
    wl = W.config5(moe=True)
    m = wl.moe
    ids = torch.from_numpy(m.topk_ids).cuda()
    perm = nv.moe_permute(ids, m.experts, row_align=ALIGN)
    xq = nv.quantize(to_dev(m.x))
    a = nv.moe_gather_quantized(xq, perm["gather"], perm["offsets"])
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    rperm = orc.moe_permute(m.topk_ids, m.experts, ALIGN, capacity=perm["capacity"])
    rx = orc.quantize(m.x)
    return dict(m=m, perm=perm, a=a, rperm=rperm, rx=rx)


def test_permute_rollout(nv, rollout):
    got, ref = rollout["perm"], rollout["rperm"]
    assert np.array_equal(host(got["offsets"]), ref["offsets"])
    assert np.array_equal(host(got["gather"]), ref["gather"])
    assert np.array_equal(host(got["dst"]), ref["dst"])
    assert int(ref["offsets"][-1]) >= 65536 * 8


def test_gather_quantized_rollout(nv, orc, rollout):
    """Row r of the layout = the oracle's quantization of token gather[r]; pad
    rows are zero; the swizzled scales of the whole layout match."""
    a, rx, g = rollout["a"], rollout["rx"], rollout["rperm"]["gather"]
    valid = g >= 0
    H = rollout["m"].hidden
    q_ref = np.zeros((g.size, H // 2), np.uint8)
    q_ref[valid] = rx["q"][g[valid]]
    sf_ref = np.zeros((g.size, H // 16), np.uint8)
    sf_ref[valid] = rx["sf"][g[valid]]
    s_ref = np.zeros(g.size, np.float32)
    s_ref[valid] = rx["s"][g[valid]]
    gq = host(a["q"])
    bad = np.argwhere(gq != q_ref)
    assert bad.size == 0, f"{len(bad)} packed bytes differ, first {bad[:5].tolist()}"
    assert np.array_equal(host(a["s"]).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(host(a["sf"]), orc.sf_swizzle(sf_ref))


def _expert_samples(rng, r0, r1, gather, N):
    """Sampled (row, column) pairs of one expert's valid rows: random ones plus
    the first and last valid row and the first and last column."""
    rows = np.nonzero(gather[r0:r1] >= 0)[0]
    mi = np.concatenate([rng.choice(rows, SAMPLES_PER_EXPERT), rows[[0, -1, -1, 0]]])
    ni = np.concatenate([rng.integers(0, N, SAMPLES_PER_EXPERT), [0, N - 1, 0, N - 1]])
    return mi, ni


def _grouped_every_expert(nv, orc, a_gpu, tokens_ref, perm, rperm, w_bits, N, K, seed):
    """Run the grouped GEMM on the GPU layout a_gpu and compare sampled outputs
    of every expert with the exact products of the oracle's quantized tokens
    (tokens_ref, indexed by source token) and the oracle's quantized weight rows."""
    E = w_bits.shape[0]
    wq = nv.quantize_experts(to_dev(w_bits.reshape(E * N, K)).reshape(E, N, K))
    y = nv.grouped_gemm(a_gpu, perm["offsets"], E, wq["q"], wq["sf"], wq["s"], N, K)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    off, g = rperm["offsets"], rperm["gather"]
    used = int(off[E])
    yb = host(y[:used])
    rng = np.random.default_rng(seed)
    checked = 0
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        mi, ni = _expert_samples(rng, r0, r1, g, N)
        toks = g[r0 + mi]
        ar = dict(q=tokens_ref["q"][toks], sf=tokens_ref["sf"][toks], s=tokens_ref["s"][toks])
        br = orc.quantize(w_bits[e][ni])
        idx = np.arange(mi.size)
        yref, absy = orc.gemm_exact_sampled(ar, br, idx, idx)
        got = W.bf16_bits_to_float(yb[r0 + mi, ni]).astype(np.float64)
        check_gemm(got, yref, absy, K, f"expert {e}")
        pad = g[r0:r1] < 0
        assert not yb[r0:r1][pad].any(), f"expert {e}: pad rows not zero"
        checked += 1
    assert checked == E
    return y


def test_grouped_fc1_rollout_every_expert(nv, orc, rollout):
    m = rollout["m"]
    _grouped_every_expert(nv, orc, rollout["a"], rollout["rx"], rollout["perm"], rollout["rperm"], m.w1,
                          2 * m.ffn, m.hidden, seed=51)


def test_grouped_swiglu_rollout(nv, rollout):
    """fc1 with the SwiGLU epilogue at full size: the same bits as the grouped
    GEMM followed by the SwiGLU kernel (each checked against the oracle here and
    in the MoE tests), rows past the layout zero."""
    m = rollout["m"]
    E, F, H = m.experts, m.ffn, m.hidden
    wq = nv.quantize_experts(to_dev(m.w1.reshape(E * 2 * F, H)).reshape(E, 2 * F, H))
    off = rollout["perm"]["offsets"]
    y1 = nv.grouped_gemm(rollout["a"], off, E, wq["q"], wq["sf"], wq["s"], 2 * F, H)
    ref = nv.swiglu_quantize(y1, F, row_count=off[E:], want_h=True)
    del y1
    h = nv.grouped_gemm_swiglu(rollout["a"], off, E, wq["q"], wq["sf"], wq["s"], F, H)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    used = int(rollout["rperm"]["offsets"][-1])
    assert torch.equal(h[:used].view(torch.int16), ref["h"][:used].view(torch.int16))
    assert not h[used:].view(torch.int16).any()


def test_grouped_fc2_rollout_every_expert(nv, orc, rollout):
    """fc2 on seeded expert inputs h [65536, 768] (quantized once, copied to the
    layout by the same permutation)."""
    m = rollout["m"]
    h = W.random_bf16_bits(52, (m.tokens, m.ffn), exp_lo=118, exp_hi=128)
    hq = nv.moe_gather_quantized(nv.quantize(to_dev(h)), rollout["perm"]["gather"], rollout["perm"]["offsets"])
    _grouped_every_expert(nv, orc, hq, orc.quantize(h), rollout["perm"], rollout["rperm"], m.w2,
                          m.hidden, m.ffn, seed=53)


def test_swiglu_quantize_rollout(nv, orc, rollout):
    """The fc2-input stage on a seeded full-size fc1 output [capacity, 1536]
    with the layout's used-row count on the device: sampled rows checked,
    every row past the count zero."""
    m = rollout["m"]
    F = m.ffn
    cap = rollout["perm"]["capacity"]
    off = rollout["perm"]["offsets"]
    used = int(rollout["rperm"]["offsets"][-1])
    y1 = W.random_bf16_bits(54, (cap, 2 * F), exp_lo=118, exp_hi=130)
    got = nv.swiglu_quantize(to_dev(y1), F, row_count=off[m.experts:], want_h=True)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    rng = np.random.default_rng(55)
    rows = np.unique(np.concatenate([rng.integers(0, used, 4096), [0, used - 1]]))
    h_ref = orc.swiglu(y1[rows], F)
    hb = host(got["h"][torch.from_numpy(rows).cuda()])
    hg = W.bf16_bits_to_float(hb).astype(np.float64)
    hr = W.bf16_bits_to_float(h_ref).astype(np.float64)
    assert np.all(np.abs(hg - hr) <= bf16_ulp(hr)), "h differs by more than one bf16 ulp"
    # rows whose h agrees exactly quantize bit-exactly (the fused quantize is
    # the row quantizer's code); h itself is within one bf16 ulp (silu's
    # evaluation is not fixed by the pages)
    same = np.all(hb == h_ref, axis=1)
    print(f"swiglu rollout: {same.mean():.4f} of sampled rows with h bit-exact, "
          f"{np.mean(hb != h_ref):.2e} of elements one ulp apart")
    assert np.mean(hb != h_ref) < 1e-4 and same.mean() > 0.95
    ref = orc.quantize(h_ref)
    sel = torch.from_numpy(rows[same]).cuda()
    assert np.array_equal(host(got["q"][sel]), ref["q"][same])
    assert np.array_equal(host(got["s"][sel]).view(np.uint32), ref["s"][same].view(np.uint32))
    sf_rm = orc.sf_unswizzle(host(got["sf"]), cap, F // 16)
    assert np.array_equal(sf_rm[rows[same]], ref["sf"][same])
    assert not got["q"][used:].any() and not got["s"][used:].any() and not got["h"][used:].any()
    assert not sf_rm[used:].any()


def test_combine_rollout(nv, orc, rollout):
    """Unpermute + weighted combine of a seeded full-size fc2 output; sampled
    tokens bit-exact against the oracle's binary32 slot-order reduction."""
    m = rollout["m"]
    cap = rollout["perm"]["capacity"]
    y2 = W.random_bf16_bits(56, (cap, m.hidden), exp_lo=116, exp_hi=128)
    w = W.topk_weights(4, m.tokens, m.topk)
    dst = rollout["rperm"]["dst"]
    yd = torch.from_numpy(y2.view(np.int16)).cuda().view(torch.bfloat16)
    out = nv.moe_combine(yd, rollout["perm"]["dst"], torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    assert nv.nvfp4_get_device_status() == 0
    rng = np.random.default_rng(57)
    toks = np.unique(np.concatenate([rng.integers(0, m.tokens, 4096), [0, m.tokens - 1]]))
    want = orc.moe_combine(y2, dst[toks], w[toks])
    got = host(out[torch.from_numpy(toks).cuda()])
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} differ, first {bad[:5].tolist()}"
