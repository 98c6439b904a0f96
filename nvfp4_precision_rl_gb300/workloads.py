"""Seeded synthetic inputs for the five workloads (host numpy, bf16 bits as uint16).

This module holds none of the method's arithmetic: it only draws random
tensors and rounds them to bfloat16.  Both the CUDA library's tests/bench and
the CPU oracle consume exactly these bytes, so the two sides never depend on
each other's random number generators.

Shapes follow the Qwen3 learner/rollout workloads the pages measure: sequence
length 4096 with micro-batch 1, Qwen3-4B MLP up-projection, Qwen3-30B-A3B MoE
experts (hidden 2048, expert FFN 768, 128 experts, top-8), as in
"Native NVFP4 RL destabilizes late in training: miniTE lifts full learner
updates to about 1.33-1.37x BF16" (LMSYS summary, "Perspective": sequence 4096,
micro-batch 1) and "Towards Blackwell-Native 8-bit and 4-bit RL" ("Experimental
setup": Qwen3-30B-A3B).  The pages' datasets are not used; these synthetic
tensors stand in for the activations of those runs.

Every workload uses numpy's PCG64 with seed (index - 1); draws happen in the
order written below.
"""
from dataclasses import dataclass, field

import numpy as np
import torch


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bits (round to nearest even, via torch's CPU cast)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_float(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng, shape, std=1.0):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


@dataclass
class MoEInputs:
    tokens: int
    hidden: int
    ffn: int
    experts: int
    topk: int
    x: np.ndarray            # [tokens, hidden] bf16 bits
    topk_ids: np.ndarray     # [tokens, topk] int32
    w1: np.ndarray = None    # [experts, 2*ffn, hidden] bf16 bits (gate rows first, then up)
    w2: np.ndarray = None    # [experts, hidden, ffn] bf16 bits


@dataclass
class Workload:
    name: str
    seed: int
    x: np.ndarray = None           # [M, K] bf16 bits
    w: np.ndarray = None           # [N, K] bf16 bits
    column_copy: bool = False
    modes: tuple = ("per_token",)
    seq_lens: np.ndarray = None
    moe: MoEInputs = None
    meta: dict = field(default_factory=dict)


def route_topk(rng, tokens, experts, topk):
    """Top-k experts of softmax(logits), logits ~ N(0,1).  Softmax is monotone,
    so the top-k of the softmax is the top-k of the logits; ties (probability
    zero for continuous draws) go to the lower expert id, slots in descending
    logit order."""
    logits = rng.standard_normal(size=(tokens, experts), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")
    return np.ascontiguousarray(order[:, :topk].astype(np.int32))


def topk_weights(seed, tokens, topk):
    """Seeded combine weights [tokens, topk] (float32): positive, summing to about
    one per token, in descending order like slots taken in descending logit
    order.  Synthetic input data for the weighted combine."""
    rng = np.random.default_rng(np.random.PCG64(1000 + seed))
    e = np.exp(rng.standard_normal(size=(tokens, topk)))
    e = -np.sort(-e, axis=1)
    return np.ascontiguousarray((e / e.sum(axis=1, keepdims=True)).astype(np.float32))


def moe_inputs(rng, tokens, hidden=2048, ffn=768, experts=128, topk=8, weights=True):
    topk_ids = route_topk(rng, tokens, experts, topk)
    x = to_bf16_bits(_normal(rng, (tokens, hidden)))
    m = MoEInputs(tokens, hidden, ffn, experts, topk, x, topk_ids)
    if weights:
        m.w1 = np.empty((experts, 2 * ffn, hidden), np.uint16)
        m.w2 = np.empty((experts, hidden, ffn), np.uint16)
        for e in range(experts):
            m.w1[e] = to_bf16_bits(_normal(rng, (2 * ffn, hidden), 0.02))
        for e in range(experts):
            m.w2[e] = to_bf16_bits(_normal(rng, (hidden, ffn), 0.02))
    return m


def config1():
    """Single linear: X [128, 512] ~ N(0,1) with 2 outlier channels x20,
    W [256, 512] ~ N(0, 0.02)."""
    rng = np.random.Generator(np.random.PCG64(0))
    x = _normal(rng, (128, 512))
    cols = rng.choice(512, size=2, replace=False)
    x[:, cols] *= np.float32(20.0)
    w = _normal(rng, (256, 512), 0.02)
    return Workload("single_linear_128x256x512", 0, to_bf16_bits(x), to_bf16_bits(w),
                    meta=dict(outlier_cols=cols.tolist()))


def config2(M=4096, N=9728, K=2560):
    """Qwen3-4B MLP up-projection: X [4096, 2560] ~ N(0,1) with Bernoulli(0.001)
    entries x30, W [9728, 2560] ~ N(0, 0.02); row- and column-wise copies of X."""
    rng = np.random.Generator(np.random.PCG64(1))
    x = _normal(rng, (M, K))
    hit = rng.random(size=(M, K), dtype=np.float32) < np.float32(0.001)
    x[hit] *= np.float32(30.0)
    w = _normal(rng, (N, K), 0.02)
    return Workload(f"qwen3_4b_up_proj_{M}x{N}x{K}", 1, to_bf16_bits(x), to_bf16_bits(w),
                    column_copy=True)


def config3(tokens=4096, weights=True):
    """Qwen3-30B-A3B MoE experts: 4096 tokens, hidden 2048, 128 experts, top-8
    of softmax(N(0,1) logits); fc1 [128, 1536, 2048], fc2 [128, 2048, 768] ~ N(0, 0.02)."""
    rng = np.random.Generator(np.random.PCG64(2))
    moe = moe_inputs(rng, tokens, weights=weights)
    return Workload(f"qwen3_30b_a3b_moe_{tokens}tok_128e_top8", 2, moe=moe)


def config4(M=16384, N=4096, K=4096):
    """Heavy tails: X [16384, 4096] Student-t(3) = N(0,1)/sqrt(chi2_3/3), 8 channels
    x50; W [4096, 4096] ~ N(0, 0.02); per-token and per-tensor outer scales."""
    rng = np.random.Generator(np.random.PCG64(3))
    z = _normal(rng, (M, K))
    chi2 = rng.chisquare(3.0, size=(M, K)).astype(np.float32)
    x = z / np.sqrt(chi2 / np.float32(3.0))
    cols = rng.choice(K, size=8, replace=False)
    x[:, cols] *= np.float32(50.0)
    w = _normal(rng, (N, K), 0.02)
    return Workload(f"heavy_tail_{M}x{N}x{K}", 3, to_bf16_bits(x), to_bf16_bits(w),
                    modes=("per_token", "per_tensor"), meta=dict(outlier_cols=cols.tolist()))


def varlen_lengths(rng, n_seq=64, lo=256, hi=8192, total=65536):
    """64 lengths ~ U[256, 8192] rescaled to sum to 65536: L' = max(256,
    floor(L * total / sum L)), the remainder added to (or taken from) the longest."""
    L = rng.integers(lo, hi + 1, size=n_seq)
    Ls = np.maximum(lo, np.floor(L * total / L.sum()).astype(np.int64))
    Ls[np.argmax(Ls)] += total - Ls.sum()
    return Ls


def config5(M=65536, N=6144, K=2048, moe=True, moe_weights=True):
    """Variable-length rollout batch: 64 sequences concatenated to 65536 tokens,
    X ~ N(0,1) times a per-sequence LogNormal(0,1) scale, fused QKV W [6144, 2048];
    plus the MoE experts of config 3 at this token count."""
    rng = np.random.Generator(np.random.PCG64(4))
    lens = varlen_lengths(rng, total=M)
    scale = rng.lognormal(0.0, 1.0, size=lens.size).astype(np.float32)
    x = _normal(rng, (M, K))
    x *= np.repeat(scale, lens)[:, None]
    w = _normal(rng, (N, K), 0.02)
    wl = Workload(f"varlen_rollout_{M}x{N}x{K}", 4, to_bf16_bits(x), to_bf16_bits(w), seq_lens=lens)
    if moe:
        wl.moe = moe_inputs(rng, M, weights=moe_weights)
    return wl


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def small_matrix(seed, M, K, dist="normal", std=1.0, outlier_cols=0, outlier_scale=20.0):
    """Small seeded matrices for parity tests (several tiles and a ragged tail)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if dist == "normal":
        x = _normal(rng, (M, K), std)
    elif dist == "student_t3":
        x = _normal(rng, (M, K)) / np.sqrt(rng.chisquare(3.0, size=(M, K)).astype(np.float32) / 3)
    elif dist == "lognormal_rows":
        x = _normal(rng, (M, K)) * rng.lognormal(0.0, 1.0, size=(M, 1)).astype(np.float32)
    else:
        raise ValueError(dist)
    if outlier_cols:
        cols = rng.choice(K, size=outlier_cols, replace=False)
        x[:, cols] *= np.float32(outlier_scale)
    return to_bf16_bits(x)


def init_data_class(kind, seed, M, K):
    """The four quantizer test classes named on the pages' bit-exact contract
    ("random", "boundary", "zeros", "maxes").  "boundary" places elements on
    E2M1 rounding ties of a block whose scale is exactly representable, and
    block amaxes on E4M3 ties; "maxes" fills rows with +-bf16 max."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if kind == "random":
        return to_bf16_bits(_normal(rng, (M, K)))
    if kind == "zeros":
        z = np.zeros((M, K), np.float32)
        z[rng.random((M, K)) < 0.5] = -0.0   # signed zeros too
        return to_bf16_bits(z)
    if kind == "maxes":
        bmax = np.float32(3.3895313892515355e38)
        sign = np.where(rng.random((M, K)) < 0.5, np.float32(-1), np.float32(1))
        return to_bf16_bits(sign * bmax)
    if kind == "boundary":
        # Row r: element 0 is the row amax 2688 * 2^e, so the per-token scale is
        # exactly 2^e.  Every other block is one of two tie cases:
        #  (a) a power-of-two block scale sb with block amax 6 * sb * S and the
        #      other elements at E2M1 rounding ties (0.25, 0.75, ... 5) * sb * S;
        #  (b) a block amax of 6 * S * mid, mid the midpoint of two adjacent
        #      E4M3 values, so the block scale itself lands on an E4M3 tie.
        e2m1_ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
        e4m3 = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
        x = np.zeros((M, K), np.float32)
        for r in range(M):
            S = np.float32(2.0) ** int(rng.integers(-20, 10))
            x[r, :16] = _normal(rng, 16) * np.float32(100.0) * S
            x[r, 0] = np.float32(2688.0) * S
            for b in range(1, K // 16):
                if rng.random() < 0.5:
                    sb = np.float32(2.0) ** int(rng.integers(-9, 8))
                    v = rng.choice(e2m1_ties, size=16) * np.where(rng.random(16) < 0.5, -1, 1)
                    v[int(rng.integers(0, 16))] = np.float32(6.0)
                    x[r, 16 * b:16 * b + 16] = v.astype(np.float32) * sb * S
                else:
                    i = int(rng.integers(0, 126))
                    mid = np.float32(0.5) * (e4m3[i] + e4m3[i + 1])
                    v = np.clip(_normal(rng, 16) * np.float32(2.0), -5.4, 5.4) * mid * S
                    v[int(rng.integers(0, 16))] = np.float32(6.0) * mid * S
                    x[r, 16 * b:16 * b + 16] = v
        return to_bf16_bits(x)
    raise ValueError(kind)


def random_bf16_bits(seed, shape, exp_lo=119, exp_hi=131):
    """Seeded bf16 bit patterns: random sign and 7-bit mantissa, biased exponent
    uniform in [exp_lo, exp_hi] (magnitudes 2^(exp_lo - 127) .. 2^(exp_hi - 126)).
    A fast stand-in, at full size, for the bf16 outputs of an expert GEMM."""
    rng = np.random.Generator(np.random.PCG64(seed))
    r = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    e = rng.integers(exp_lo, exp_hi + 1, size=shape, dtype=np.uint16)
    return (r & np.uint16(0x807F)) | (e << np.uint16(7))
