#!/usr/bin/env python
"""Benchmark of the per-token NVFP4 W4A4 linear-layer hot path on GB300.

One step = one pass of the whole hot path over the variable-length rollout
batch (65,536 tokens, hidden 2048), the largest workload that fits one GPU:
  dense half: per-token quantize of X [65536, 2048] and per-row quantize of the
      fused QKV weight W [6144, 2048] (one launch), block-scaled W4A4 GEMM
      -> Y bf16 [65536, 6144];
  MoE half (Qwen3-30B-A3B experts at the same token count: 128 experts, top-8,
      524,288 routed rows): routing permute, per-token quantize of the tokens,
      copy of their quantized rows into the per-expert layout, grouped fc1
      (2048 -> 2 x 768) with SwiGLU in its epilogue (h bf16), per-token quantize
      of h, grouped fc2 (768 -> 2048), unpermute + weighted combine -> bf16
      [65536, 2048].
The expert and QKV weights are quantized once (fixed within a step) for the
MoE half; the dense half quantizes its weight every step.

value    = algorithmic GEMM FLOP of the step (2 M N K dense + 2 R (2F H + F H)
           grouped over the routed rows R; padding not counted), all ranks,
           / device step time (CUDA events on the launching stream around the
           step's per-stage graphs; L2 flushed before every step).
e2e      = the same metric through the library calls with HOST buffers: the
           step's inputs copied in from pinned memory and both outputs copied
           back inside the timed region.
roofline = the kernel that takes most of the step (the grouped GEMM with the
           SwiGLU epilogue, fc1): its algorithmic FLOP over its CUDA-event
           duration inside the timed region, against the FP4 peak derived from
           the measured bf16 peak (x6, the 13.5/2.25 nominal ratio); fraction
           of 9 PF beside it.
Sections: the dense GEMM and the quantizer of the same workload per call, the
heavy-tailed 16384x4096x4096 workload (per-token and per-tensor), the Qwen3-4B
learner layer (column copy, backward GEMMs, dequantize, MXFP8) and the MoE
step at 4096 tokens.

--impl reference times the CPU oracle (oracle/) on a bounded sample of the
same workload on the host cores.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A4 GEMM TFLOPS (% of 9 PF FP4) and per-token quantize GB/s (% of HBM)"
WORKLOAD = "varlen_rollout_65536x6144x2048+moe_65536tok_128e_top8"
PAGES_FP4_PF = 9.0          # the target denominator named with the metric
NOMINAL_FP4_PF = 13.5       # the pages' B300 dense FP4 row
BF16_TO_FP4 = 13.5 / 2.25   # nominal dense FP4 / BF16 ratio
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
SOAK_S = 0.6                # untimed replays before the timed steps (clocks settle)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sections", default="c4,c2,c3",
                    help="extra sections after the headline: c4, c2, c3 (comma list, or 'none')")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sections-only", action="store_true",
                    help="run only the extra sections (small cases for profiling); prints their JSON")
    ap.add_argument("--moe-row-align", type=int, default=256, choices=[128, 256],
                    help="expert segment alignment of the MoE layout (256: one pair tile per slot)")
    ap.add_argument("--moe-section-tokens", type=int, default=4096,
                    help="tokens of the MoE section (c3): 4096, or more for a compute-bound case "
                         "small enough to profile")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value, device, world):
    """Largest value of a per-rank float across ranks (the step time the job sees)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, seconds_max):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / seconds_max


def measured_peaks():
    """HBM GB/s, bf16 burst and sustained TFLOP/s: the measured file's figures,
    else (file or key missing, or unreadable) the fallback measurement."""
    fallback = (6800.0, 1900.0, 1700.0)
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        vals = (d.get("hbm_gbs"), d.get("bf16_tflops"), d.get("bf16_tflops_sustained"))
    except (OSError, ValueError):
        return fallback + ("fallback",)
    if all(isinstance(v, (int, float)) and v > 0 for v in vals):
        return vals + ("measured",)
    return fallback + ("fallback",)


def code_sha(path):
    """sha256 of a source file's code: // comments, trailing blanks and blank
    lines removed, so a comment edit does not orphan counters taken on it."""
    with open(path) as f:
        lines = [ln.split("//", 1)[0].rstrip() for ln in f.read().splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def kernel_traffic(kernel_sha, workload, launch):
    """DRAM bytes of one launch from the committed ncu summary, if it was taken
    on the current kernel source and this workload."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("gemm_cu_code_sha256") != kernel_sha:
        return None
    entry = d.get("launches", {}).get(f"{workload}:{launch}")
    return None if entry is None else entry.get("dram_bytes")


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU works."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.2)   # the sampler is up before the work starts

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [ln.strip().split(",") for ln in self.tmp.read().splitlines() if ln.strip()]
        os.unlink(self.tmp.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: power well above idle (the first samples may precede the work)
        p = np.array(power)
        busy = p > max(300.0, 0.5 * float(p.max()))
        sm_busy = np.array(sm)[busy] if busy.any() else np.array(sm)
        return {"sm_mhz": float(np.median(sm_busy)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": int(busy.sum()),
                "power_w_max": float(p.max())}


# ----------------------------------------------------------------------------
# Steps built from the library calls
# ----------------------------------------------------------------------------

class Stage:
    """One library call of a step: its name, the call, and how many of the
    library's kernels it launches."""

    def __init__(self, name, fn, kernels, flop=0.0, nbytes=0.0, kernel=None):
        self.name, self.fn, self.kernels = name, fn, kernels
        self.flop, self.kernel = flop, kernel
        # algorithmic bytes: a number, or (read, write)
        self.rbytes, self.wbytes = nbytes if isinstance(nbytes, tuple) else (nbytes, 0.0)
        self.nbytes = self.rbytes + self.wbytes


def bf16_dev(torch, bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


class DenseLayer:
    """X [M, K] and W [N, K] quantized in one launch (optionally with X's
    column-wise copy), then Y = X W^T through the W4A4 GEMM."""

    def __init__(self, ops, torch, dev, stream, x, w, column_copy):
        self.ops, self.stream = ops, stream
        self.M, self.K = x.shape
        self.N = w.shape[0]
        self.x, self.w = x, w
        M, N, K = self.M, self.N, self.K
        u8 = torch.uint8
        self.qx = dict(rows=M, cols=K, q=torch.empty((M, K // 2), dtype=u8, device=dev),
                       sf=torch.empty(ops.nvfp4_sf_bytes(M, K), dtype=u8, device=dev),
                       s=torch.empty(M, dtype=torch.float32, device=dev))
        self.qw = dict(rows=N, cols=K, q=torch.empty((N, K // 2), dtype=u8, device=dev),
                       sf=torch.empty(ops.nvfp4_sf_bytes(N, K), dtype=u8, device=dev),
                       s=torch.empty(N, dtype=torch.float32, device=dev))
        self.column_copy = column_copy
        self.qcol = self.sfcol = self.scol = None
        if column_copy:
            self.qcol = torch.empty((K, M // 2), dtype=u8, device=dev)
            self.sfcol = torch.empty(ops.nvfp4_sf_bytes(K, M), dtype=u8, device=dev)
            self.scol = torch.empty(1, dtype=torch.float32, device=dev)
        self.wsb = ops.nvfp4_quantize_workspace_bytes()
        self.ws = torch.empty(self.wsb, dtype=u8, device=dev)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

    def quant_rw(self):
        """Algorithmic (read, write) bytes of the quantize call: read 2 B per
        element, write 0.5 B codes + 1/16 B scales per element + 4 B per row
        (X and W rows); the column copy writes another 0.5 + 1/16 B per element
        of X + 4 B."""
        M, N, K = self.M, self.N, self.K
        r = (M + N) * K * 2
        w = (M + N) * K * (0.5 + 1 / 16) + (M + N) * 4
        if self.column_copy:
            w += M * K * (0.5 + 1 / 16) + 4
        return r, w

    def quant_bytes(self):
        return sum(self.quant_rw())

    def flop(self):
        return 2.0 * self.M * self.N * self.K

    def quantize(self, x=None):
        o = self.ops
        o.nvfp4_quantize_per_token_pair(self.x if x is None else x, self.M, self.K, self.qx["q"], self.qx["sf"],
                                        self.qx["s"], self.qcol, self.sfcol, self.scol, self.w, self.N, self.K,
                                        self.qw["q"], self.qw["sf"], self.qw["s"], self.K, self.ws, self.wsb,
                                        self.stream)

    def gemm(self, y=None):
        y = self.y if y is None else y
        self.ops.nvfp4_gemm(self.qx["q"], self.qx["sf"], self.qx["s"], self.M, self.qw["q"], self.qw["sf"],
                            self.qw["s"], self.N, self.K, y, self.N, self.stream)

    def stages(self):
        return [Stage("quantize_x_w", self.quantize, 2 if self.column_copy else 1, nbytes=self.quant_rw(),
                      kernel="quant_rows_staged_kernel"),
                Stage("gemm", self.gemm, 1, flop=self.flop(), kernel="nvfp4_gemm_pair_kernel<0, 0, 0>")]


class MoELayer:
    """The routed-expert step: permute, per-token quantize of the tokens, copy of
    their quantized rows into the per-expert layout, grouped fc1 with the SwiGLU
    epilogue, per-token quantize of h, grouped fc2, unpermute + weighted combine."""

    def __init__(self, ops, torch, dev, stream, moe, combine_weights, align):
        self.ops, self.stream = ops, stream
        T, H, F, E, k = moe.tokens, moe.hidden, moe.ffn, moe.experts, moe.topk
        self.T, self.H, self.F, self.E, self.k, self.align = T, H, F, E, k, align
        u8, i32 = torch.uint8, torch.int32
        self.x = bf16_dev(torch, moe.x, dev)
        self.ids = torch.from_numpy(moe.topk_ids).to(dev)
        w1 = bf16_dev(torch, moe.w1, dev)
        self.w1 = ops.quantize_experts(w1, stream=stream)
        del w1
        w2 = bf16_dev(torch, moe.w2, dev)
        self.w2 = ops.quantize_experts(w2, stream=stream)
        del w2
        cap = ops.nvfp4_moe_capacity(T, k, E, align)
        self.cap = cap
        self.off = torch.empty(E + 1, dtype=i32, device=dev)
        self.gather = torch.empty(cap, dtype=i32, device=dev)
        self.dst = torch.empty((T, k), dtype=i32, device=dev)
        self.pws_b = ops.nvfp4_moe_permute_workspace_bytes(T, k, E)
        self.pws = torch.empty(max(self.pws_b, 256), dtype=u8, device=dev)
        self.xq = dict(q=torch.empty((T, H // 2), dtype=u8, device=dev),
                       sf=torch.empty(ops.nvfp4_sf_bytes(T, H), dtype=u8, device=dev),
                       s=torch.empty(T, dtype=torch.float32, device=dev))
        self.a = dict(q=torch.empty((cap, H // 2), dtype=u8, device=dev),
                      sf=torch.empty(ops.nvfp4_sf_bytes(cap, H), dtype=u8, device=dev),
                      s=torch.empty(cap, dtype=torch.float32, device=dev))
        self.h = torch.empty((cap, F), dtype=torch.bfloat16, device=dev)
        self.hq = dict(q=torch.empty((cap, F // 2), dtype=u8, device=dev),
                       sf=torch.empty(ops.nvfp4_sf_bytes(cap, F), dtype=u8, device=dev),
                       s=torch.empty(cap, dtype=torch.float32, device=dev))
        self.y2 = torch.empty((cap, H), dtype=torch.bfloat16, device=dev)
        self.cw = torch.from_numpy(combine_weights).to(dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.used_rows = None

    def routed(self):
        return self.T * self.k

    def flops(self):
        R, H, F = self.routed(), self.H, self.F
        return 2.0 * R * H * 2 * F, 2.0 * R * F * H

    def stage_bytes(self):
        """Algorithmic (read, write) bytes per stage over the ROUTED rows
        (padding rows of the aligned layout are not counted): each must move
        these at least once."""
        T, H, F, E, k, R = self.T, self.H, self.F, self.E, self.k, self.routed()
        qrow_h = H // 2 + H // 16 + 4      # codes + block scales + S of one quantized row
        qrow_f = F // 2 + F // 16 + 4
        w1 = E * (2 * F) * (H // 2 + H // 16 + 4)
        w2 = E * H * (F // 2 + F // 16 + 4)
        return {
            "permute": (T * k * 4, R * 4 + T * k * 4 + (E + 1) * 4),
            "quantize_tokens": (T * H * 2, T * qrow_h),
            # each token's quantized row is read once from HBM (its other k - 1
            # reads hit L2) and written to its k routed rows
            "gather_quantized": (T * qrow_h, R * qrow_h),
            "grouped_fc1_swiglu": (R * qrow_h + w1, R * F * 2),
            "quantize_h": (R * F * 2, R * qrow_f),
            "grouped_fc2": (R * qrow_f + w2, R * H * 2),
            "combine": (R * H * 2 + T * k * 8, T * H * 2),
        }

    def stages(self, x=None, ids=None, out=None):
        o, s = self.ops, self.stream
        T, H, F, E, k, cap, al = self.T, self.H, self.F, self.E, self.k, self.cap, self.align
        x = self.x if x is None else x
        ids = self.ids if ids is None else ids
        out = self.out if out is None else out
        fl1, fl2 = self.flops()
        nb = self.stage_bytes()
        return [
            Stage("permute", lambda: o.nvfp4_moe_permute(ids, T, k, E, al, self.off, self.gather, cap, self.dst,
                                                         self.pws, self.pws_b, s), 3, nbytes=nb["permute"],
                  kernel="perm_count/scan/scatter_kernel"),
            # per-token quantization of the tokens once, then their rows copied to the
            # routed layout (equal, bit for bit, to quantizing the gathered rows)
            Stage("quantize_tokens", lambda: o.nvfp4_quantize_per_token(
                x, T, H, H, None, T, o.PER_TOKEN, self.xq["q"], self.xq["sf"], self.xq["s"], stream=s), 1,
                nbytes=nb["quantize_tokens"], kernel="quant_rows_staged_kernel"),
            Stage("gather_quantized", lambda: o.nvfp4_moe_gather_quantized(
                self.xq["q"], self.xq["sf"], self.xq["s"], T, H, self.gather, cap, self.off, E, self.a["q"],
                self.a["sf"], self.a["s"], s), 1, nbytes=nb["gather_quantized"], kernel="gather_quantized_kernel"),
            # fc1 (gate + up) with SwiGLU in the GEMM epilogue: h [cap, F] bf16,
            # rows past the layout zero; then per-token quantization of h
            Stage("grouped_fc1_swiglu", lambda: o.nvfp4_grouped_gemm_swiglu(
                self.a["q"], self.a["sf"], self.a["s"], cap, self.off, E, self.w1["q"], self.w1["sf"],
                self.w1["s"], F, H, self.h, s), 1, flop=fl1, nbytes=nb["grouped_fc1_swiglu"],
                kernel="nvfp4_gemm_pair_kernel<1, 1, 0>"),
            Stage("quantize_h", lambda: o.nvfp4_quantize_per_token(
                self.h, cap, F, F, None, cap, o.PER_TOKEN, self.hq["q"], self.hq["sf"], self.hq["s"], stream=s), 1,
                nbytes=nb["quantize_h"], kernel="quant_row_pairs_kernel (768 columns)"),
            Stage("grouped_fc2", lambda: o.nvfp4_grouped_gemm(
                self.hq["q"], self.hq["sf"], self.hq["s"], cap, self.off, E, self.w2["q"], self.w2["sf"],
                self.w2["s"], H, F, self.y2, s), 1, flop=fl2, nbytes=nb["grouped_fc2"],
                kernel="nvfp4_gemm_pair_kernel<1, 0, 0>"),
            Stage("combine", lambda: o.nvfp4_moe_combine(self.y2, cap, H, self.dst, self.cw, T, k, H, out, H, s),
                  1, nbytes=nb["combine"], kernel="combine_kernel"),
        ]


# ----------------------------------------------------------------------------
# Timing
# ----------------------------------------------------------------------------

class Timer:
    def __init__(self, torch, stream, flush):
        self.torch, self.stream, self.flush = torch, stream, flush

    def ev(self):
        return self.torch.cuda.Event(enable_timing=True)

    def capture(self, fns):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for fn in fns:
                fn()
        torch.cuda.synchronize()
        return g

    def staged(self, graphs, steps):
        """steps x (L2 flush, then the per-stage graphs with an event before,
        between and after them); returns [steps, stages] ms."""
        runs = []
        for _ in range(steps):
            self.flush.zero_()
            evs = [self.ev() for _ in range(len(graphs) + 1)]
            for i, g in enumerate(graphs):
                evs[i].record(self.stream)
                g.replay()
            evs[-1].record(self.stream)
            runs.append(evs)
        self.torch.cuda.synchronize()
        return np.array([[e[i].elapsed_time(e[i + 1]) for i in range(len(graphs))] for e in runs])

    def one_graph(self, g, steps):
        ts = []
        for _ in range(steps):
            self.flush.zero_()
            e0, e1 = self.ev(), self.ev()
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
            ts.append((e0, e1))
        self.torch.cuda.synchronize()
        return np.array([a.elapsed_time(b) for a, b in ts])

    def soak(self, g, seconds):
        """Replays g (untimed) for about `seconds` of GPU time; returns the replays."""
        self.torch.cuda.synchronize()
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < seconds:
            for _ in range(4):
                g.replay()
                n += 1
            self.torch.cuda.synchronize()
        return n

    def rotating(self, fns, reps, min_seconds=0.0):
        """Per-call time of fns (distinct buffer sets, together larger than L2)
        captured back to back in one graph: the graph's time / len(fns), mean over
        reps (at least min_seconds of replays)."""
        for _ in range(2):
            for fn in fns:
                fn()
        self.torch.cuda.synchronize()
        g = self.capture(fns)
        ts = []
        t0 = time.perf_counter()
        while len(ts) < reps or time.perf_counter() - t0 < min_seconds:
            self.flush.zero_()
            e0, e1 = self.ev(), self.ev()
            e0.record(self.stream)
            g.replay()
            e1.record(self.stream)
            self.torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / len(fns))
        return float(np.mean(ts)), len(ts)


def one_way_bandwidth(torch, dev, flush):
    """Read-only and write-only DRAM bandwidth (GB/s) on this GPU, measured with
    CUDA events: a sum over and a fill of 2 GB as 8-byte words (best of five;
    a fill of bytes or 2-byte words is store-issue-bound at ~4 TB/s)."""
    buf = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
    words = buf.view(torch.int64)

    def best(fn):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return buf.numel() / (min(ts) * 1e-3) / 1e9
    rd = best(lambda: words.sum())
    wr = best(lambda: words.fill_(1))
    del buf, words
    torch.cuda.empty_cache()
    return rd, wr


def rot_note(n):
    return f"{n} calls per graph over {n} buffer sets (> L2), per-call average"


# ----------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    from nvfp4_precision_rl_gb300 import _build
    from nvfp4_precision_rl_gb300 import ops
    from nvfp4_precision_rl_gb300 import workloads as W

    _build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    # one side stream for everything: the library calls are stream-ordered and
    # allocation-free, so each stage is captured once into a CUDA graph and replayed
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    tm = Timer(torch, stream, flush)
    hbm_gbs, bf16_burst, bf16_sust, peak_src = measured_peaks()
    fp4_burst, fp4_sust = bf16_burst * BF16_TO_FP4, bf16_sust * BF16_TO_FP4
    launches = 0

    def check_status(where):
        st = ops.nvfp4_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {where}: {ops.STATUS_NAMES.get(st)}")

    if args.sections_only:
        return run_sections(args, torch, ops, W, dev, stream, tm, fp4_burst, hbm_gbs, check_status, world)
    # ------------------------------------------------------------------ headline
    wl = W.config5()
    x5 = bf16_dev(torch, wl.x, dev)
    w5 = bf16_dev(torch, wl.w, dev)
    dense = DenseLayer(ops, torch, dev, stream, x5, w5, column_copy=False)
    moe = MoELayer(ops, torch, dev, stream, wl.moe, W.topk_weights(4, wl.moe.tokens, wl.moe.topk),
                   args.moe_row_align)
    stages = dense.stages() + moe.stages()
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        for st in stages:
            st.fn()
    torch.cuda.synchronize()
    check_status("after warm-up")
    moe.used_rows = int(moe.off[moe.E].item())
    graphs = [tm.capture([st.fn]) for st in stages]
    g_step = tm.capture([st.fn for st in stages])

    clocks = Clocks(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    soak_n = tm.soak(g_step, SOAK_S)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    seg = tm.staged(graphs, args.steps)                       # [steps, stages] ms, the timed region
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    launches += args.steps * sum(st.kernels for st in stages)
    if world > 1:
        torch.distributed.barrier()
    t_step = seg.sum(axis=1)
    ms_step = float(t_step.mean())
    ms_step_max = max_over_ranks(ms_step, dev, world)
    flop_step = sum(st.flop for st in stages)
    value = job_throughput(flop_step, world, ms_step_max * 1e-3) / 1e12
    t_one = tm.one_graph(g_step, args.steps)
    launches += args.steps * sum(st.kernels for st in stages)
    seg_ms = seg.mean(axis=0)
    kernels_ms = {st.name if i >= 2 else f"dense_{st.name}": round(float(seg_ms[i]), 5)
                  for i, st in enumerate(stages)}

    # the roofline kernel: the library kernel with the most time in the step
    by_kernel = {}
    for i, st in enumerate(stages):
        k = by_kernel.setdefault(st.kernel, {"ms": 0.0, "flop": 0.0, "bytes": 0.0, "launches": []})
        k["ms"] += float(seg_ms[i])
        k["flop"] += st.flop
        k["bytes"] += st.nbytes
        k["launches"].append(st.name)
    top = max(by_kernel, key=lambda n: by_kernel[n]["ms"])
    tk = by_kernel[top]
    sha = code_sha(os.path.join(ROOT, "nvfp4_precision_rl_gb300", "csrc", "gemm.cu"))
    if tk["flop"] > 0:
        ach = tk["flop"] / (tk["ms"] * 1e-3) / 1e12
        traffic = [kernel_traffic(sha, "c5", n) for n in tk["launches"]]
        roof = {"kernel": top, "bound": "tensor", "achieved": round(ach, 1), "peak": round(fp4_sust, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp4_sust, 4),
                "frac_of_9pf": round(ach / (PAGES_FP4_PF * 1000), 4),
                "frac_of_13p5pf": round(ach / (NOMINAL_FP4_PF * 1000), 4),
                "frac_of_burst_peak": round(ach / fp4_burst, 4),
                "peak_basis": f"{peak_src} bf16 sustained {bf16_sust} TFLOP/s x {BF16_TO_FP4:g} (FP4/BF16 "
                              f"nominal): the kernel is timed inside a {ms_step:.2f} ms step",
                "traffic": (None if any(t is None for t in traffic) else round(sum(traffic) / len(traffic))),
                "launches_per_step": tk["launches"],
                "kernel_ms_per_launch": round(tk["ms"] / len(tk["launches"]), 5),
                "timing": "CUDA events between the step's per-stage graphs inside the timed region",
                "sm_mhz_median": clk.get("sm_mhz")}
        per = {}
        for i, st in enumerate(stages):
            if st.kernel == top:
                a = st.flop / (seg_ms[i] * 1e-3) / 1e12
                per[st.name] = {"ms": round(float(seg_ms[i]), 5), "tflops": round(a, 1),
                                "frac_of_9pf": round(a / (PAGES_FP4_PF * 1000), 4),
                                "hbm_gbs_on_algorithmic_bytes": round(st.nbytes / (seg_ms[i] * 1e-3) / 1e9, 1),
                                "hbm_frac": round(st.nbytes / (seg_ms[i] * 1e-3) / 1e9 / hbm_gbs, 4)}
        roof["per_launch"] = per
    else:
        ach = tk["bytes"] / (tk["ms"] * 1e-3) / 1e9
        roof = {"kernel": top, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_gbs, "unit": "GB/s",
                "frac": round(ach / hbm_gbs, 4), "traffic": None}

    # ---- per-stage rooflines of the step (algorithmic bytes / FLOP over routed rows)
    rw_bw = one_way_bandwidth(torch, dev, flush)
    stage_report = {}
    for i, st in enumerate(stages):
        ms = float(seg_ms[i])
        r = {"ms": round(ms, 5)}
        if st.nbytes:
            r["gbs"] = round(st.nbytes / (ms * 1e-3) / 1e9, 1)
            r["hbm_frac"] = round(st.nbytes / (ms * 1e-3) / 1e9 / hbm_gbs, 4)
            # DRAM time bound: the slowest of the reads at the measured read-only
            # rate, the writes at the write-only rate (~4 TB/s on this part) and
            # all bytes at the copy rate
            bound_ms = max(st.rbytes / rw_bw[0], st.wbytes / rw_bw[1], st.nbytes / hbm_gbs) / 1e9 * 1e3
            r["rw_bound_ms"] = round(bound_ms, 5)
            r["frac_of_rw_bound"] = round(bound_ms / ms, 4)
        if st.flop:
            r["tflops"] = round(st.flop / (ms * 1e-3) / 1e12, 1)
            r["frac_of_9pf"] = round(st.flop / (ms * 1e-3) / 1e12 / (PAGES_FP4_PF * 1000), 4)
        stage_report[st.name if i >= 2 else f"dense_{st.name}"] = r

    # ---- per-call: the dense GEMM and the quantizer of the same workload, alone
    ROT = 3
    qsets = []
    for i in range(ROT):
        xi = x5 if i == 0 else x5.clone()
        d = DenseLayer(ops, torch, dev, stream, xi, w5, column_copy=False)
        qsets.append(d)
    t_q, n_q = tm.rotating([d.quantize for d in qsets], args.steps)
    for d in qsets:
        d.quantize()
    clocks_g = Clocks(local_rank)
    clocks_g.start()
    t_g, n_g = tm.rotating([d.gemm for d in qsets], args.steps, min_seconds=0.6)
    clk_g = clocks_g.stop()
    launches += ROT * (n_q + n_g)
    q_gbs = dense.quant_bytes() / (t_q * 1e-3) / 1e9
    g_tf = dense.flop() / (t_g * 1e-3) / 1e12
    dense_percall = {
        "gemm": {"ms": round(t_g, 5), "tflops": round(g_tf, 1), "frac": round(g_tf / fp4_burst, 4),
                 "frac_of_9pf": round(g_tf / (PAGES_FP4_PF * 1000), 4),
                 "peak": round(fp4_burst, 1),
                 "peak_basis": f"{peak_src} bf16 burst {bf16_burst} x {BF16_TO_FP4:g}",
                 "traffic": kernel_traffic(sha, "c5", "gemm"),
                 "timing": rot_note(ROT) + f", {n_g} replays over >= 0.6 s", "clocks": clk_g},
        "quantize_x_w": {"ms": round(t_q, 5), "gbs": round(q_gbs, 1), "frac": round(q_gbs / hbm_gbs, 4),
                         "bytes": int(dense.quant_bytes()), "timing": rot_note(ROT)},
    }
    del qsets

    # ---- end to end through the library calls with host buffers
    e2e = run_e2e(args, torch, ops, dev, stream, wl, dense, moe, world)
    e2e_value = job_throughput(flop_step, world, e2e["ms_per_step"] * 1e-3) / 1e12
    launches += e2e.pop("launches")
    check_status("after the headline")

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 (e2m1 x e4m3) -> fp32 acc -> bf16",
        "data": "synthetic (seeded numpy PCG64; Qwen3-shaped rollout activations, QKV and expert weights)",
        "config": ref_config(),
        "run": {"parallelism": f"dp{world} (independent batches, no collective)",
                "moe_routed_rows": moe.routed(), "moe_layout_rows": moe.used_rows, "moe_row_align": moe.align,
                "l2": "flushed (512 MB write) before every timed step",
                "launch": "each library call captured once as a CUDA graph; the timed step replays them "
                          "in order with CUDA events between them",
                "gemm_flop_per_step": flop_step},
        "e2e": dict(e2e, value=round(e2e_value, 2), unit="TFLOP/s"),
        "roofline": roof,
        "kernels_ms": kernels_ms,
        "stages": stage_report,
        "one_graph_ms_per_step": round(float(t_one.mean()), 5),
        "hbm_one_way_gbs": {"read": round(rw_bw[0], 1), "write": round(rw_bw[1], 1),
                            "how": "sum over / fill of 2 GB as int64 words, best of five, CUDA events"},
        "quantize": {"gbs": dense_percall["quantize_x_w"]["gbs"], "frac": dense_percall["quantize_x_w"]["frac"],
                     "hbm_peak_gbs": hbm_gbs, "peak_basis": f"{peak_src} copy bandwidth",
                     "what": "per-token X [65536, 2048] rows + W [6144, 2048] rows, one launch, per call",
                     "in_step_gbs": stage_report["dense_quantize_x_w"]["gbs"],
                     "moe_tokens_in_step_gbs": stage_report["quantize_tokens"]["gbs"]},
        "dense": dense_percall,
        "clocks": clk,
        "clocks_note": f"sampled every 50 ms from before a {SOAK_S} s untimed soak of the step graph "
                       f"({soak_n} replays) through the timed steps",
        "wall_s_timed_loop": round(t_wall, 3),
    }
    del dense, moe, stages, graphs, g_step, x5, w5, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    sections = run_sections(args, torch, ops, W, dev, stream, tm, fp4_burst, hbm_gbs, check_status, world)
    launches += sections.pop("gpu_launches")
    result.update(sections)
    result["gpu_launches"] = launches
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline()
    if world > 1:
        torch.distributed.destroy_process_group()
    return result


def run_sections(args, torch, ops, W, dev, stream, tm, fp4_burst, hbm_gbs, check_status, world):
    """The extra workloads (per call): heavy-tailed, Qwen3-4B learner layer,
    MoE step at 4096 tokens."""
    out, launches = {}, 0
    secs = [s for s in args.sections.split(",") if s and s != "none"]
    if "c4" in secs:
        out["heavy_tail_16384x4096x4096"], n = section_c4(torch, ops, W, dev, tm, args, fp4_burst, hbm_gbs)
        launches += n
    if "c2" in secs:
        out["qwen3_4b_up_proj_4096x9728x2560"], n = section_c2(torch, ops, W, dev, stream, tm, args, fp4_burst,
                                                               hbm_gbs)
        launches += n
    if "c3" in secs:
        out[f"qwen3_30b_a3b_moe_{args.moe_section_tokens}tok"], n = section_c3(torch, ops, W, dev, stream, tm, args,
                                                                               hbm_gbs)
        launches += n
    check_status("after the sections")
    out["gpu_launches"] = launches
    if args.sections_only and world > 1:
        torch.distributed.destroy_process_group()
    return out


def run_e2e(args, torch, ops, dev, stream, wl, dense, moe, world):
    """The step through the library calls with host buffers, pipelined as a
    rollout loop runs it: copy-in, compute and copy-out on three streams with
    double-buffered device staging, so step i's output copies and step i+1's
    input copies overlap the compute; every step still moves its own inputs in
    and its own outputs out inside the timed window."""
    pin = lambda t: t.pin_memory()  # noqa: E731
    x_host = pin(torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16))
    mx_host = pin(torch.from_numpy(wl.moe.x.view(np.int16)).view(torch.bfloat16))
    ids_host = pin(torch.from_numpy(wl.moe.topk_ids))
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    xs = [torch.empty_like(dense.x) for _ in range(2)]
    mxs = [torch.empty_like(moe.x) for _ in range(2)]
    idss = [torch.empty_like(moe.ids) for _ in range(2)]
    ys = [torch.empty_like(dense.y) for _ in range(2)]
    outs = [torch.empty_like(moe.out) for _ in range(2)]
    yh = [pin(torch.empty(dense.y.shape, dtype=torch.bfloat16)) for _ in range(2)]
    oh = [pin(torch.empty(moe.out.shape, dtype=torch.bfloat16)) for _ in range(2)]
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def pipe_step(i):
        b = i % 2
        if i >= 2:
            s_in.wait_event(comp_done[b])          # the staging of step i-2 was read
        with torch.cuda.stream(s_in):
            xs[b].copy_(x_host, non_blocking=True)
            mxs[b].copy_(mx_host, non_blocking=True)
            idss[b].copy_(ids_host, non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if i >= 2:
            stream.wait_event(out_done[b])         # the outputs of step i-2 are on the host
        dense.quantize(xs[b])
        dense.gemm(ys[b])
        for st in moe.stages(x=mxs[b], ids=idss[b], out=outs[b]):
            st.fn()
        comp_done[b].record(stream)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            yh[b].copy_(ys[b], non_blocking=True)
            oh[b].copy_(outs[b], non_blocking=True)
        out_done[b].record(s_out)

    w = max(3, args.warmup)
    for i in range(w):
        pipe_step(i)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(s_in)
    for i in range(args.steps):
        pipe_step(i + 2 * w)
    p1.record(s_out)
    torch.cuda.synchronize()
    ms = max_over_ranks(p0.elapsed_time(p1) / args.steps, dev, world)
    kern = 2 + 9
    h2d = x_host.numel() * 2 + mx_host.numel() * 2 + ids_host.numel() * 4
    d2h = yh[0].numel() * 2 + oh[0].numel() * 2
    return {"ms_per_step": round(ms, 5), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "mode": "pipelined: copy-in / compute / copy-out streams, double-buffered staging, no L2 flush "
                    "(the step's working set exceeds L2); the dense Y and the MoE output copied back every step",
            "launches": (w + args.steps) * kern}


def section_c4(torch, ops, W, dev, tm, args, fp4_burst, hbm_gbs):
    """Heavy-tailed X [16384, 4096] (Student-t, 8 outlier channels), W [4096, 4096]:
    per-token and per-tensor quantize per call, and the GEMM per call."""
    wl = W.config4()
    x = bf16_dev(torch, wl.x, dev)
    w = bf16_dev(torch, wl.w, dev)
    M, K = x.shape
    N = w.shape[0]
    ROT = 3
    xs = [x] + [x.clone() for _ in range(ROT - 1)]
    layers = [DenseLayer(ops, torch, dev, tm.stream, xi, w, column_copy=False) for xi in xs]
    t_pair, n1 = tm.rotating([d.quantize for d in layers], args.steps)
    # per-tensor outer scale on X (a tensor-wide amax pass, then the rows)
    outs = [ops.quantize(xi, mode="per_tensor") for xi in xs]
    wsb = ops.nvfp4_quantize_workspace_bytes()
    wss = [torch.empty(wsb, dtype=torch.uint8, device=dev) for _ in xs]

    def per_tensor(xi, o, ws):
        ops.nvfp4_quantize_per_token(xi, M, K, K, None, M, ops.PER_TENSOR, o["q"], o["sf"], o["s"],
                                     workspace=ws, workspace_bytes=wsb, stream=tm.stream)

    def per_token(xi, o):
        ops.nvfp4_quantize_per_token(xi, M, K, K, None, M, ops.PER_TOKEN, o["q"], o["sf"], o["s"],
                                     stream=tm.stream)
    t_pt, n2 = tm.rotating([lambda a=a, o=o, s=s: per_tensor(a, o, s) for a, o, s in zip(xs, outs, wss)],
                           args.steps)
    t_tok, n3 = tm.rotating([lambda a=a, o=o: per_token(a, o) for a, o in zip(xs, outs)], args.steps)
    for d in layers:
        d.quantize()
    t_g, n4 = tm.rotating([d.gemm for d in layers], args.steps)
    xb = M * K * (2 + 0.5 + 1 / 16) + M * 4
    pair_b = layers[0].quant_bytes()
    fl = 2.0 * M * N * K
    res = {
        "workload": f"heavy_tail_{M}x{N}x{K}",
        "quantize_x_w_per_token": {"ms": round(t_pair, 5), "gbs": round(pair_b / (t_pair * 1e-3) / 1e9, 1),
                                   "frac": round(pair_b / (t_pair * 1e-3) / 1e9 / hbm_gbs, 4)},
        "quantize_x_per_token": {"ms": round(t_tok, 5), "gbs": round(xb / (t_tok * 1e-3) / 1e9, 1),
                                 "frac": round(xb / (t_tok * 1e-3) / 1e9 / hbm_gbs, 4)},
        "quantize_x_per_tensor": {"ms": round(t_pt, 5), "gbs": round(xb / (t_pt * 1e-3) / 1e9, 1),
                                  "frac": round(xb / (t_pt * 1e-3) / 1e9 / hbm_gbs, 4),
                                  "note": "algorithmic bytes as per token; the kernel reads X twice "
                                          "(tensor amax, then the rows)"},
        "gemm": {"ms": round(t_g, 5), "tflops": round(fl / (t_g * 1e-3) / 1e12, 1),
                 "frac": round(fl / (t_g * 1e-3) / 1e12 / fp4_burst, 4),
                 "frac_of_9pf": round(fl / (t_g * 1e-3) / 1e12 / (PAGES_FP4_PF * 1000), 4)},
        "timing": rot_note(ROT),
    }
    n = ROT * (n1 + 2 * n2 + n3 + n4)
    del layers, outs, xs, x, w
    torch.cuda.empty_cache()
    return res, n


def section_c2(torch, ops, W, dev, stream, tm, args, fp4_burst, hbm_gbs):
    """The Qwen3-4B learner layer (X [4096, 2560], W [9728, 2560]): quantize
    with X's column-wise copy + GEMM, the backward GEMMs on the column-wise
    copies, NVFP4 dequantization and the MXFP8 copies of X."""
    wl = W.config2()
    x = bf16_dev(torch, wl.x, dev)
    w = bf16_dev(torch, wl.w, dev)
    M, K = x.shape
    N = w.shape[0]
    ROT = 8
    layer = DenseLayer(ops, torch, dev, stream, x, w, column_copy=True)
    st = layer.stages()
    for _ in range(3):
        for s in st:
            s.fn()
    torch.cuda.synchronize()
    graphs = [tm.capture([s.fn]) for s in st]
    seg = tm.staged(graphs, args.steps).mean(axis=0)
    layers = [layer] + [DenseLayer(ops, torch, dev, stream, x.clone(), w, column_copy=True)
                        for _ in range(ROT - 1)]
    t_q, n1 = tm.rotating([d.quantize for d in layers], args.steps)
    for d in layers:
        d.quantize()
    t_g, n2 = tm.rotating([d.gemm for d in layers], args.steps)
    fl = layer.flop()
    qb = layer.quant_bytes()
    res = {"workload": f"qwen3_4b_up_proj_{M}x{N}x{K}",
           "step_ms": round(float(seg.sum()), 5),
           "step_tflops": round(fl / (seg.sum() * 1e-3) / 1e12, 1),
           "kernels_ms": {"quantize_x_rows_cols_w": round(float(seg[0]), 5), "gemm": round(float(seg[1]), 5)},
           "quantize_x_rows_cols_w": {"ms": round(t_q, 5), "gbs": round(qb / (t_q * 1e-3) / 1e9, 1),
                                      "frac": round(qb / (t_q * 1e-3) / 1e9 / hbm_gbs, 4)},
           "gemm": {"ms": round(t_g, 5), "tflops": round(fl / (t_g * 1e-3) / 1e12, 1),
                    "frac": round(fl / (t_g * 1e-3) / 1e12 / fp4_burst, 4),
                    "frac_of_9pf": round(fl / (t_g * 1e-3) / 1e12 / (PAGES_FP4_PF * 1000), 4)},
           "timing": rot_note(ROT)}
    n = args.steps * 3 + ROT * (2 * n1 + n2)
    # NVFP4 -> bf16 dequantization of the quantized activation
    dq_out = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(ROT)]
    t_dq, m = tm.rotating([lambda d=d, o=o: ops.nvfp4_dequantize(d.qx["q"], d.qx["sf"], d.qx["s"], 1, M, K, o, K,
                                                                 stream) for d, o in zip(layers, dq_out)],
                          args.steps)
    n += ROT * m
    dq_b = M * K * (0.5 + 1 / 16) + M * 4 + M * K * 2
    res["dequantize"] = {"ms": round(t_dq, 5), "gbs": round(dq_b / (t_dq * 1e-3) / 1e9, 1),
                         "frac": round(dq_b / (t_dq * 1e-3) / 1e9 / hbm_gbs, 4)}
    del dq_out
    # MXFP8: 1x32 row copy + 32x1 column copy of X, then the row copy back to bf16
    mx_out = [ops.mxfp8_quantize(d.x, column_copy=True) for d in layers]
    t_mq, m1 = tm.rotating([lambda d=d, o=o: ops.nvfp4_mxfp8_quantize(d.x, M, K, K, o["q"], o["sf"], o["q_col"],
                                                                      o["sf_col"], stream)
                            for d, o in zip(layers, mx_out)], args.steps)
    ymx = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(ROT)]
    t_md, m2 = tm.rotating([lambda o=o, yo=yo: ops.nvfp4_mxfp8_dequantize(o["q"], o["sf"], M, K, yo, K, stream)
                            for o, yo in zip(mx_out, ymx)], args.steps)
    n += ROT * (2 * m1 + m2)
    mq_b = M * K * 2 + 2 * (M * K + M * K / 32)
    md_b = M * K + M * K / 32 + M * K * 2
    res["mxfp8"] = {"quantize_row_col_ms": round(t_mq, 5), "quantize_gbs": round(mq_b / (t_mq * 1e-3) / 1e9, 1),
                    "quantize_frac": round(mq_b / (t_mq * 1e-3) / 1e9 / hbm_gbs, 4),
                    "dequantize_ms": round(t_md, 5), "dequantize_gbs": round(md_b / (t_md * 1e-3) / 1e9, 1),
                    "dequantize_frac": round(md_b / (t_md * 1e-3) / 1e9 / hbm_gbs, 4)}
    del mx_out, ymx
    # backward GEMMs on the column-wise copies: dgrad dX = dY W, wgrad dW = dY^T X
    dy = bf16_dev(torch, W.small_matrix(77, M, N, std=1e-3), dev)
    qdy = ops.quantize(dy, column_copy=True)
    qwc = ops.quantize(w, column_copy=True)
    qxc = ops.quantize(x, column_copy=True)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    bw = [lambda: ops.gemm_dgrad(qdy, qwc, out=dx, stream=stream),
          lambda: ops.gemm_wgrad(qdy, qxc, out=dw, stream=stream)]
    for _ in range(3):
        for fn in bw:
            fn()
    torch.cuda.synchronize()
    gbw = [tm.capture([fn]) for fn in bw]
    t_bw = tm.staged(gbw, args.steps).mean(axis=0)
    n += 2 * args.steps
    res["backward"] = {"dgrad_ms": round(float(t_bw[0]), 5), "wgrad_ms": round(float(t_bw[1]), 5),
                       "dgrad_tflops": round(fl / (t_bw[0] * 1e-3) / 1e12, 1),
                       "wgrad_tflops": round(fl / (t_bw[1] * 1e-3) / 1e12, 1),
                       "shapes": {"dgrad": [M, K, N], "wgrad": [N, K, M]}}
    del layers, layer, qdy, qwc, qxc, dx, dw, dy, x, w
    torch.cuda.empty_cache()
    return res, n


def section_c3(torch, ops, W, dev, stream, tm, args, hbm_gbs):
    """The MoE expert step of the Qwen3-30B-A3B workload at 4096 tokens (or
    --moe-section-tokens)."""
    wl = W.config3(tokens=args.moe_section_tokens)
    moe = MoELayer(ops, torch, dev, stream, wl.moe, W.topk_weights(2, wl.moe.tokens, wl.moe.topk),
                   args.moe_row_align)
    st = moe.stages()
    for _ in range(max(3, args.warmup)):
        tm.flush.zero_()
        for s in st:
            s.fn()
    torch.cuda.synchronize()
    moe.used_rows = int(moe.off[moe.E].item())
    graphs = [tm.capture([s.fn]) for s in st]
    g_all = tm.capture([s.fn for s in st])
    seg = tm.staged(graphs, args.steps).mean(axis=0)
    tot = float(tm.one_graph(g_all, args.steps).mean())
    fl1, fl2 = moe.flops()
    stages = {}
    for i, s in enumerate(st):
        r = {"ms": round(float(seg[i]), 5), "gbs": round(s.nbytes / (seg[i] * 1e-3) / 1e9, 1),
             "hbm_frac": round(s.nbytes / (seg[i] * 1e-3) / 1e9 / hbm_gbs, 4)}
        if s.flop:
            r["tflops"] = round(s.flop / (seg[i] * 1e-3) / 1e12, 1)
        stages[s.name] = r
    res = {"workload": f"qwen3_30b_a3b_moe_{wl.moe.tokens}tok_128e_top8 (hidden 2048, expert ffn 768)",
           "ms_per_step": round(tot, 5), "stage_graphs_ms": round(float(seg.sum()), 5),
           "tflops": round((fl1 + fl2) / (tot * 1e-3) / 1e12, 1),
           "routed_rows": moe.routed(), "layout_rows": moe.used_rows, "row_align": moe.align,
           "stages": stages,
           "bytes_basis": "algorithmic bytes over routed rows (padding of the aligned layout not counted)"}
    n = 2 * args.steps * sum(s.kernels for s in st)
    del moe, st, graphs, g_all
    torch.cuda.empty_cache()
    return res, n


# ----------------------------------------------------------------------------
# CPU oracle timings (baseline and the reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(wl, rows_x, rows_w, nthreads):
    """One bounded sample of the step on the oracle: quantize rows_x rows of X
    and rows_w rows of W, then their exact W4A4 product.  Returns (flop, s)."""
    import oracle
    K = wl.x.shape[1]
    t0 = time.perf_counter()
    a = oracle.quantize(wl.x[:rows_x], nthreads=nthreads)
    b = oracle.quantize(wl.w[:rows_w], nthreads=nthreads)
    oracle.gemm_exact(a, b, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return 2.0 * rows_x * rows_w * K, dt


RX, RW = 256, 2048


def sample_workload():
    """The dense half of the headline workload, without generating the MoE half
    (the oracle sample reads only X and W)."""
    from nvfp4_precision_rl_gb300 import workloads as W
    return W.config5(moe=False)


def cpu_baseline(target_s=12.0):
    wl = sample_workload()
    cores = os.cpu_count() or 1
    flop, dt = oracle_sample(wl, RX, RW, cores)
    reps = max(1, int(target_s / max(dt, 1e-3)))
    tot_f, tot_t = 0.0, 0.0
    for _ in range(min(reps, 400)):
        f, t = oracle_sample(wl, RX, RW, cores)
        tot_f += f
        tot_t += t
    return {"value": round(tot_f / tot_t / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"quantize {RX} rows of X and {RW} rows of W of the 65,536x6,144x2,048 workload "
                      f"(per-token), exact int64 W4A4 product {RX}x{RW}x2048; {min(reps, 400)} repetitions, "
                      f"{tot_t:.1f} s"}


def ref_config():
    return {"workload": WORKLOAD, "M_tokens": 65536, "N": 6144, "K": 2048, "sequences": 64,
            "lengths": "U[256, 8192] rescaled to sum 65,536",
            "moe": {"experts": 128, "topk": 8, "hidden": 2048, "expert_ffn": 768},
            "scale_mode": "per_token", "column_copy": False}


def run_reference(args):
    wl = sample_workload()
    cores = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle_sample(wl, RX, RW, cores)
    flops, times = 0.0, []
    for _ in range(args.steps):
        f, t = oracle_sample(wl, RX, RW, cores)
        flops = f
        times.append(t)
    ms = float(np.mean(times)) * 1e3
    value = flops / (ms * 1e-3) / 1e12
    sample = (f"per step: quantize {RX} rows of X and {RW} rows of W (per-token) of the workload, exact int64 "
              f"W4A4 product {RX}x{RW}x2048 on {cores} host threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64 exact / f64",
        "data": "synthetic (seeded numpy PCG64)",
        "config": ref_config(),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    result = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
