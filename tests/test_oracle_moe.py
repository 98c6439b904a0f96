"""Pins for the oracle's MoE routing permute and SwiGLU.

Permute: the contiguous per-expert layout with device-side metadata ("miniTE
report", section "Transformer Engine path optimisation": contiguous layouts,
device-side metadata, grouped GEMM), each expert's segment padded to a multiple
of 128 rows.  Pinned against numpy's stable argsort and invariants.

SwiGLU: silu(gate) * up between the MoE fc1 and fc2 ("Towards Blackwell-Native
8-bit and 4-bit RL", "Parallelism and tensor-conversion contract": gate and up
projections fused into one GEMM).  Pinned against float64 numpy on exact inputs
and, at chosen points across the gate's range, against 60-digit decimal
arithmetic rounded to bfloat16 on integers.
"""
import numpy as np

from nvfp4_precision_rl_gb300 import workloads as W


def _topk(seed, T, E, k):
    return W.route_topk(np.random.default_rng(seed), T, E, k)


def test_permute_vs_stable_argsort(orc):
    for T, E, k, align in [(1, 4, 1, 128), (37, 8, 2, 16), (300, 16, 4, 128), (1000, 128, 8, 128)]:
        ids = _topk(T, T, E, k)
        d = orc.moe_permute(ids, E, align)
        flat = ids.ravel()
        counts = np.bincount(flat, minlength=E)
        padded = -(-counts // align) * align
        off = np.concatenate([[0], np.cumsum(padded)])
        assert np.array_equal(d["offsets"], off)
        order = np.argsort(flat, kind="stable")          # pairs (t, j) grouped by expert
        rank = np.empty_like(order)
        rank[order] = np.arange(order.size)
        start = np.concatenate([[0], np.cumsum(counts)])[flat]
        want_dst = off[flat] + (rank - start)
        assert np.array_equal(d["dst"].ravel(), want_dst)
        want_gather = np.full(d["capacity"], -1, np.int64)
        want_gather[want_dst] = np.arange(flat.size) // k
        assert np.array_equal(d["gather"], want_gather)


def test_permute_invariants(orc):
    ids = _topk(7, 4096, 128, 8)
    d = orc.moe_permute(ids, 128, 128)
    off, g = d["offsets"], d["gather"]
    assert np.all(off % 128 == 0) and np.all(np.diff(off) >= 0)
    assert (g >= 0).sum() == 4096 * 8
    for e in range(128):
        seg = g[off[e]:off[e + 1]]
        real = seg[seg >= 0]
        assert np.all(np.diff(real) >= 0)                 # ascending token order
        assert np.all(seg[len(real):] == -1)              # padding at the end
        assert np.all((ids[real] == e).any(axis=1))
    assert d["capacity"] >= off[-1]


def test_gather_quantize_commutes(orc):
    """quantize(gather(X)) == gather(quantize(X)) byte for byte: per-token
    scales make a routed copy of a token identical to the token itself."""
    x = W.small_matrix(71, 300, 256)
    ids = _topk(72, 300, 16, 4)
    d = orc.moe_permute(ids, 16, 128)
    gq = orc.quantize(x, gather=d["gather"])
    full = orc.quantize(x)
    real = d["gather"] >= 0
    assert np.array_equal(gq["q"][real], full["q"][d["gather"][real]])
    assert np.array_equal(gq["sf"][real], full["sf"][d["gather"][real]])
    assert not gq["q"][~real].any()


def test_permute_rejects_bad_ids(orc):
    import pytest
    ids = np.array([[0, 5]], np.int32)
    with pytest.raises(ValueError):
        orc.moe_permute(ids, 4, 128)


def test_swiglu_vs_float64(orc):
    rng = np.random.default_rng(73)
    rows, F = 50, 96
    y1 = W.to_bf16_bits((rng.standard_normal((rows, 2 * F)) * 3).astype(np.float32))
    h = orc.swiglu(y1, F)
    yf = W.bf16_bits_to_float(y1).astype(np.float64)
    g, u = yf[:, :F], yf[:, F:]
    ref = g / (1.0 + np.exp(-g)) * u
    hf = W.bf16_bits_to_float(h).astype(np.float64)
    # bf16 nearest: within half a bf16 ulp of the float64 value
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-38))) - 7)
    assert np.all(np.abs(hf - ref) <= ulp / 2 * (1 + 1e-12))


def _bf16_nearest_bits(v):
    """Bits of the bfloat16 nearest to the real number v (a Decimal), ties to
    even, computed on integers: v = m 2^e with m in [2^7, 2^8) for normals."""
    from decimal import Decimal
    if v == 0:
        return 0x8000 if v.is_signed() else 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    # a in [1, 2): value = a 2^e; subnormals (e < -126) keep fewer bits
    frac_bits = 7 if e >= -126 else 7 - (-126 - e)
    scaled = a * (Decimal(2) ** frac_bits)
    q = int(scaled)
    rem = scaled - q
    if rem > Decimal("0.5") or (rem == Decimal("0.5") and q % 2 == 1):
        q += 1
    if e >= -126:
        if q == 256:                       # rounded up to the next binade
            q, e = 128, e + 1
        assert e <= 127, "overflow is not exercised here"
        return sign | ((e + 127) << 7) | (q - 128)
    return sign | q                        # subnormal: exponent field 0


def test_swiglu_high_precision_points(orc):
    """The oracle's h against silu(g) u evaluated with 60-digit decimal
    arithmetic (its own exp) and rounded to bfloat16 on integers, across the
    gate's range: exp(-g) near overflow, silu(g) far below 1, large and small
    up-projection values."""
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    gates = [-90.0, -88.5, -50.0, -20.0, -3.5, -1.0, -0.125, 0.0, 0.125, 1.0, 3.5, 20.0, 90.0]
    ups = [1.0, -3.0, 1000.0, 2.0 ** -60]
    F = len(gates)
    y1 = np.zeros((len(ups), 2 * F), np.float32)
    y1[:, :F] = gates
    y1[:, F:] = np.array(ups, np.float32)[:, None]
    bits = W.to_bf16_bits(y1)
    assert np.array_equal(W.bf16_bits_to_float(bits), y1), "test points must be bfloat16 values"
    h = orc.swiglu(bits, F)
    for i, u in enumerate(ups):
        for j, g in enumerate(gates):
            gd, ud = Decimal(g), Decimal(u)
            exact = gd / (1 + (-gd).exp()) * ud
            want = _bf16_nearest_bits(exact)
            assert int(h[i, j]) == want, (g, u, hex(int(h[i, j])), hex(want))
