"""Pins for the oracle's unpermute + weighted combine after the expert GEMMs:
out[t] = bf16_rn(sum_j w[t, j] * y2[dst[t, j]]) with binary32 accumulation in slot
order ("Towards Blackwell-Native 8-bit and 4-bit RL", shared-expert section: the
routed experts' outputs pass through a high-precision weighted reduction).

Pinned by: top-1 with unit weights (the inverse of the routing permutation,
checked against numpy indexing), exact dyadic sums (small integers times powers
of two, so every partial sum is exact and equals the integer result), the
binary64 sum within the binary32 accumulation bound, the slot order (a case
where binary32 addition order changes the result), and invalid rows.
"""
import numpy as np
import torch

from nvfp4_precision_rl_gb300 import workloads as W


def _bits(f32):
    """bf16 bits of float32 values that are exact in bf16 (inputs only)."""
    a = np.asarray(f32, np.float32)
    b = a.view(np.uint32)
    assert not np.any(b & 0xFFFF), "not a bf16 value"
    return (b >> 16).astype(np.uint16)


def _bf16_rne(f32):
    """bf16 bits of float32 values, rounded by torch (nearest-even)."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(f32, np.float32))).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _val(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def test_top1_unit_weight_is_the_inverse_permutation(orc):
    rng = np.random.default_rng(3)
    T, E, H = 300, 16, 48
    ids = W.route_topk(rng, T, E, 1)
    perm = orc.moe_permute(ids, E, align=128)
    y2 = W.to_bf16_bits(rng.standard_normal((perm["capacity"], H)).astype(np.float32))
    out = orc.moe_combine(y2, perm["dst"], np.ones((T, 1), np.float32))
    assert np.array_equal(out, y2[perm["dst"].ravel()])


def test_exact_dyadic_sums(orc):
    rng = np.random.default_rng(4)
    T, K, H, R = 64, 8, 32, 700
    y2i = rng.integers(-64, 65, size=(R, H))
    wexp = rng.integers(-4, 3, size=(T, K))
    w = np.ldexp(1.0, wexp).astype(np.float32)
    dst = rng.integers(0, R, size=(T, K)).astype(np.int32)
    out = orc.moe_combine(_bits(y2i.astype(np.float32)), dst, w)
    # every term and partial sum is a multiple of 2^-4 below 2^12: exact in binary32
    want = (y2i[dst] * np.ldexp(1.0, wexp)[:, :, None]).sum(axis=1)
    assert np.array_equal(out, _bf16_rne(want))


def test_binary64_sum_within_bound(orc):
    T, K, H = 128, 8, 256
    m = W.moe_inputs(np.random.default_rng(5), T, hidden=H, experts=32, topk=K, weights=False)
    perm = orc.moe_permute(m.topk_ids, 32, align=128)
    rng = np.random.default_rng(6)
    y2 = W.to_bf16_bits(rng.standard_normal((perm["capacity"], H)).astype(np.float32))
    w = W.topk_weights(0, T, K)
    out = _val(orc.moe_combine(y2, perm["dst"], w))
    terms = w.astype(np.float64)[:, :, None] * _val(y2)[perm["dst"].reshape(T, K)]
    exact = terms.sum(axis=1)
    bound = np.abs(terms).sum(axis=1) * (2 * K) * 2.0 ** -24 + np.abs(exact) * 2.0 ** -8
    assert np.all(np.abs(out - exact) <= bound + 1e-30)


def test_slot_order(orc):
    """Binary32 addition in slot order: terms 256, -256, c (c = 1.25 * 2^-16)
    sum to c exactly; in the order 256, c, -256 the first sum rounds 256 + c to
    256 + 2^-15 (c is 0.625 of its ulp) and the result is 2^-15."""
    c = 1.25 * 2.0 ** -16
    y2 = _bits(np.array([[256.0], [-256.0], [c]], np.float32))
    w = np.ones((1, 3), np.float32)
    out = orc.moe_combine(y2, np.array([[0, 1, 2]], np.int32), w)
    assert out[0, 0] == 0x37A0            # bf16(1.25 * 2^-16)
    out = orc.moe_combine(y2, np.array([[0, 2, 1]], np.int32), w)
    assert out[0, 0] == 0x3800            # bf16(2^-15)


def test_invalid_rows_contribute_nothing(orc):
    y2 = _bits(np.array([[2.0], [3.0]], np.float32))
    out = orc.moe_combine(y2, np.array([[0, -1, 5, 1]], np.int32), np.ones((1, 4), np.float32))
    assert _val(out)[0, 0] == 5.0
