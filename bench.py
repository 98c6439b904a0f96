#!/usr/bin/env python
"""Benchmark of the per-token NVFP4 W4A4 linear-layer hot path on GB300.

One step = one pass of the dense learner path on the Qwen3-4B MLP
up-projection workload (X [4096, 2560] bf16, seq 4096 x micro-batch 1,
W [9728, 2560]):
    per-token quantize of X (row-wise + column-wise copy for the backward)
    and per-row quantize of W (one row-kernel launch over both, then the
    column-copy kernel), block-scaled W4A4 GEMM -> Y bf16 [4096, 9728].
The same run also times the MoE expert step (Qwen3-30B-A3B shapes, 4096
tokens, 128 experts, top-8): routing permute, gather-quantize, grouped fc1,
fused SwiGLU + quantize, grouped fc2 (reported under "moe").

value  = GEMM algorithmic FLOP (2 M N K, all ranks) / device step time
         (CUDA events on the launching stream; L2 flushed before every step).
e2e    = the same metric through the library calls with HOST buffers: pinned
         X copied in, Y copied out, inside the timed region.
roofline = the dominant kernel (the GEMM): achieved FLOP/s against the FP4 peak
         derived from the measured bf16 peak (x6, the 13.5/2.25 nominal ratio).

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

M, N, K = 4096, 9728, 2560
WORKLOAD = "qwen3_4b_up_proj_4096x9728x2560"
METRIC = "W4A4 GEMM TFLOPS (% of 9 PF FP4) and per-token quantize GB/s (% of HBM)"
PAGES_FP4_PF = 9.0          # the target denominator named with the metric
NOMINAL_FP4_PF = 13.5       # the pages' B300 dense FP4 row
BF16_TO_FP4 = 13.5 / 2.25   # nominal dense FP4 / BF16 ratio
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-moe", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--moe-row-align", type=int, default=256, choices=[128, 256],
                    help="expert segment alignment of the MoE layout (256: one pair tile per slot)")
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


def capture_graphs(torch, stages, stream):
    """One CUDA graph per stage of the step (captured after the eager warm-up)."""
    graphs = []
    for fn in stages:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        graphs.append(g)
    torch.cuda.synchronize()
    return graphs


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


def gemm_traffic(kernel_sha):
    """dram bytes per GEMM launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("gemm_cu_code_sha256") != kernel_sha or d.get("workload") != WORKLOAD:
        return None
    return d.get("dram_bytes_per_launch")


def code_sha(path):
    """sha256 of a source file's code: // comments, trailing blanks and blank
    lines removed, so a comment edit does not orphan counters taken on it."""
    with open(path) as f:
        lines = [ln.split("//", 1)[0].rstrip() for ln in f.read().splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
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
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


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

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    wl = W.config2()
    x = to_dev(wl.x)
    w = to_dev(wl.w)
    ws = ops.Workspace(dev)
    # outputs, allocated once
    qx = dict(rows=M, cols=K, q=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
              sf=torch.empty(ops.nvfp4_sf_bytes(M, K), dtype=torch.uint8, device=dev),
              s=torch.empty(M, dtype=torch.float32, device=dev))
    qcol = torch.empty((K, M // 2), dtype=torch.uint8, device=dev)
    sfcol = torch.empty(ops.nvfp4_sf_bytes(K, M), dtype=torch.uint8, device=dev)
    scol = torch.empty(1, dtype=torch.float32, device=dev)
    qw = dict(rows=N, cols=K, q=torch.empty((N, K // 2), dtype=torch.uint8, device=dev),
              sf=torch.empty(ops.nvfp4_sf_bytes(N, K), dtype=torch.uint8, device=dev),
              s=torch.empty(N, dtype=torch.float32, device=dev))
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    wsb = ops.nvfp4_quantize_workspace_bytes()
    wsbuf = ws.get(wsb)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def quant_xw(src):
        # X (rows + column-wise copy) and W (rows) in one row-kernel launch
        ops.nvfp4_quantize_per_token_pair(src, M, K, qx["q"], qx["sf"], qx["s"], qcol, sfcol, scol,
                                          w, N, K, qw["q"], qw["sf"], qw["s"], K, wsbuf, wsb, stream)

    def gemm():
        ops.nvfp4_gemm(qx["q"], qx["sf"], qx["s"], M, qw["q"], qw["sf"], qw["s"], N, K, y, N, stream)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    stages = [lambda: quant_xw(x), gemm]
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        for fn in stages:
            fn()
    torch.cuda.synchronize()
    st = ops.nvfp4_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {ops.STATUS_NAMES.get(st)}")
    graphs = capture_graphs(torch, stages, stream)
    # the whole step as one graph (what is timed); the per-stage graphs give the split
    (g_step,) = capture_graphs(torch, [lambda: [fn() for fn in stages]], stream)

    def step(evs=None):
        for i, g in enumerate(graphs):
            if evs:
                evs[i].record(stream)
            g.replay()
        if evs:
            evs[len(graphs)].record(stream)

    for _ in range(2):
        flush.zero_()
        step()
        flush.zero_()
        g_step.replay()
    torch.cuda.synchronize()

    clocks = Clocks(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    steps_ev = []
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()                      # L2 flush, outside the timed events
        evs = [ev(), ev()]
        evs[0].record(stream)
        g_step.replay()
        evs[1].record(stream)
        steps_ev.append(evs)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    # per-stage split: the same kernels, one graph per stage, events between
    split_ev = []
    for _ in range(args.steps):
        flush.zero_()
        evs = [ev() for _ in range(len(stages) + 1)]
        step(evs)
        split_ev.append(evs)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_step = np.array([e[0].elapsed_time(e[1]) for e in steps_ev])        # ms
    t_q = np.array([e[0].elapsed_time(e[1]) for e in split_ev])
    t_gemm = np.array([e[1].elapsed_time(e[2]) for e in split_ev])
    ms_step = float(t_step.mean())
    ms_step_max = max_over_ranks(ms_step, dev, world)
    flop = 2.0 * M * N * K
    value = job_throughput(flop, world, ms_step_max * 1e-3) / 1e12

    # ---- end to end through the library calls with host buffers ----
    x_host = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    x_stage = torch.empty_like(x)
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        x_stage.copy_(x_host, non_blocking=True)
        quant_xw(x_stage)
        gemm()
        y_host.copy_(y, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_serial = max_over_ranks(float(np.mean(e2e_ms)), dev, world)

    # the same, pipelined as a serving / training loop runs it: copy-in, compute
    # and copy-out on three streams with double-buffered staging, so step i's
    # output copy and step i+1's input copy overlap the compute; every step
    # still moves its own X in and its own Y out inside the timed window
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    xs = [torch.empty_like(x) for _ in range(2)]
    ys = [torch.empty_like(y) for _ in range(2)]
    yh = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def pipe_step(i):
        b = i % 2
        if i >= 2:
            s_in.wait_event(comp_done[b])          # xs[b] was read by step i-2
        with torch.cuda.stream(s_in):
            xs[b].copy_(x_host, non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if i >= 2:
            stream.wait_event(out_done[b])         # ys[b] of step i-2 is on the host
        quant_xw(xs[b])
        ops.nvfp4_gemm(qx["q"], qx["sf"], qx["s"], M, qw["q"], qw["sf"], qw["s"], N, K, ys[b], N, stream)
        comp_done[b].record(stream)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            yh[b].copy_(ys[b], non_blocking=True)
        out_done[b].record(s_out)

    for i in range(max(3, args.warmup)):
        pipe_step(i)
    torch.cuda.synchronize()
    p0, p1 = ev(), ev()
    p0.record(s_in)
    for i in range(args.steps):
        pipe_step(i + 2 * max(3, args.warmup))
    p1.record(s_out)
    torch.cuda.synchronize()
    e2e_step = max_over_ranks(p0.elapsed_time(p1) / args.steps, dev, world)
    e2e_value = job_throughput(flop, world, e2e_step * 1e-3) / 1e12

    hbm_gbs, bf16_burst, bf16_sust, peak_src = measured_peaks()
    fp4_peak = bf16_burst * BF16_TO_FP4
    gemm_tflops = flop / (t_gemm.mean() * 1e-3) / 1e12
    # per-token quantize of X: algorithmic bytes = read 2 B/elem + write 0.5 B codes
    # + 1/16 B scales per elem + 4 B per row; the column copy writes the same again
    qx_bytes_row = M * K * 2 + M * K * 0.5 + M * K / 16 + M * 4
    qx_bytes = qx_bytes_row + M * K * 0.5 + M * K / 16 + 4
    qw_bytes = N * K * 2 + N * K * 0.5 + N * K / 16 + N * 4
    q_gbs = (qx_bytes + qw_bytes) / (t_q.mean() * 1e-3) / 1e9
    sha = code_sha(os.path.join(ROOT, "nvfp4_precision_rl_gb300", "csrc", "gemm.cu"))

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e4m3) -> fp32 acc -> bf16",
        "data": "synthetic (seeded numpy PCG64, Qwen3-4B-shaped activations and weights)",
        "config": {"workload": WORKLOAD, "M_tokens": M, "N": N, "K": K, "seq_len": 4096,
                   "micro_batch": 1, "column_copy": True, "scale_mode": "per_token",
                   "parallelism": f"dp{world} (independent batches, no collective)",
                   "l2": "flushed (512 MB write) before every timed step",
                   "launch": "the step (quantize + GEMM) captured once as one CUDA graph and replayed; kernels_ms from one graph per stage"},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(M * K * 2), "d2h_bytes_per_step": int(M * N * 2),
                "ms_per_step": round(e2e_step, 5),
                "mode": "pipelined: copy-in / compute / copy-out streams, double-buffered staging, "
                        "no L2 flush (the step's working set exceeds L2)",
                "serial_ms_per_step": round(e2e_serial, 5),
                "serial_value": round(job_throughput(flop, world, e2e_serial * 1e-3) / 1e12, 2)},
        "roofline": {"kernel": "nvfp4_gemm_pair_kernel", "bound": "tensor",
                     "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp4_peak, 4),
                     "peak_basis": f"{peak_src} bf16 burst {bf16_burst} TFLOP/s x {BF16_TO_FP4:g} (FP4/BF16 nominal)",
                     "traffic": gemm_traffic(sha),
                     "frac_of_9pf": round(gemm_tflops / (PAGES_FP4_PF * 1000), 4),
                     "frac_of_13p5pf": round(gemm_tflops / (NOMINAL_FP4_PF * 1000), 4)},
        "kernels_ms": {"quantize_x_row_col_and_w": round(float(t_q.mean()), 5),
                       "gemm": round(float(t_gemm.mean()), 5)},
        "quantize": {"x_row_col_and_w_gbs": round(q_gbs, 1), "hbm_peak_gbs": hbm_gbs,
                     "frac": round(q_gbs / hbm_gbs, 4), "peak_basis": f"{peak_src} copy bandwidth",
                     "launches": "row kernel over X and W rows, then the X column-copy kernel"},
        "clocks": clk,
        "gpu_launches": 3 * args.steps,
        "wall_s_timed_loop": round(t_wall, 3),
    }
    # Short kernels are timed ROT calls to a graph over ROT distinct buffer sets
    # (together larger than L2), per-call average: one graph per call would add
    # the graph launch (several microseconds) to every call.
    ROT = 8

    def time_rotating(fns):
        for _ in range(2):
            for fn in fns:
                fn()
        torch.cuda.synchronize()
        (g,) = capture_graphs(torch, [lambda: [fn() for fn in fns]], stream)
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = ev(), ev()
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / len(fns))
        return float(np.mean(ts))

    rot_note = f"{ROT} calls per graph over {ROT} buffer sets (> L2), per-call average"
    # the step's quantize (X rows + column copy, W rows) per call, same method
    q_sets = []
    for _ in range(ROT):
        xi, wi = x.clone(), w.clone()
        q_sets.append(dict(x=xi, w=wi, qx=ops.quantize(xi, column_copy=True), qw=ops.quantize(wi)))

    def q_call(c):
        ops.nvfp4_quantize_per_token_pair(c["x"], M, K, c["qx"]["q"], c["qx"]["sf"], c["qx"]["s"], c["qx"]["q_col"],
                                          c["qx"]["sf_col"], c["qx"]["s_col"], c["w"], N, K, c["qw"]["q"],
                                          c["qw"]["sf"], c["qw"]["s"], K, wsbuf, wsb, stream)
    t_qrot = time_rotating([lambda c=c: q_call(c) for c in q_sets])
    result["quantize"]["per_call_ms"] = round(t_qrot, 5)
    result["quantize"]["per_call_gbs"] = round((qx_bytes + qw_bytes) / (t_qrot * 1e-3) / 1e9, 1)
    result["quantize"]["per_call_frac"] = round((qx_bytes + qw_bytes) / (t_qrot * 1e-3) / 1e9 / hbm_gbs, 4)
    result["quantize"]["per_call_timing"] = rot_note
    result["gpu_launches"] += 2 * ROT * args.steps
    # the GEMM per call, same method (the roofline's kernel time): the 8
    # quantized operand sets above, 8 output buffers
    y_sets = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(ROT)]
    t_grot = time_rotating([lambda c=c, yo=yo: ops.nvfp4_gemm(c["qx"]["q"], c["qx"]["sf"], c["qx"]["s"], M,
                                                               c["qw"]["q"], c["qw"]["sf"], c["qw"]["s"], N, K,
                                                               yo, N, stream)
                            for c, yo in zip(q_sets, y_sets)])
    g_rot = flop / (t_grot * 1e-3) / 1e12
    rf = result["roofline"]
    rf["achieved_stage_graph"] = rf["achieved"]
    rf.update({"achieved": round(g_rot, 1), "frac": round(g_rot / fp4_peak, 4),
               "frac_of_9pf": round(g_rot / (PAGES_FP4_PF * 1000), 4),
               "frac_of_13p5pf": round(g_rot / (NOMINAL_FP4_PF * 1000), 4),
               "kernel_ms": round(t_grot, 5), "timing": rot_note})
    result["gpu_launches"] += ROT * args.steps
    del q_sets, y_sets
    # NVFP4 -> bf16 dequantization of the same activation (the dequantized backward's input)
    dq_src = [dict(q=qx["q"].clone(), sf=qx["sf"].clone(), s=qx["s"].clone()) for _ in range(ROT)]
    dq_out = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(ROT)]
    dq_t = time_rotating([lambda a=a, o=o: ops.nvfp4_dequantize(a["q"], a["sf"], a["s"], 1, M, K, o, K, stream)
                          for a, o in zip(dq_src, dq_out)])
    dq_bytes = M * K * 0.5 + M * K / 16 + M * 4 + M * K * 2
    result["dequantize"] = {"ms": round(dq_t, 5), "gbs": round(dq_bytes / (dq_t * 1e-3) / 1e9, 1),
                            "frac_of_hbm": round(dq_bytes / (dq_t * 1e-3) / 1e9 / hbm_gbs, 4),
                            "shape": [M, K], "timing": rot_note}
    result["gpu_launches"] += ROT * args.steps
    # MXFP8 of the same activation: 1x32 row copy + 32x1 column copy, then the
    # row copy dequantized back to bf16
    mx_x = [x.clone() for _ in range(ROT)]
    mx_out = [ops.mxfp8_quantize(xi, column_copy=True) for xi in mx_x]
    t_mq = time_rotating([lambda xi=xi, o=o: ops.nvfp4_mxfp8_quantize(xi, M, K, K, o["q"], o["sf"], o["q_col"],
                                                                      o["sf_col"], stream)
                          for xi, o in zip(mx_x, mx_out)])
    ymx = [torch.empty((M, K), dtype=torch.bfloat16, device=dev) for _ in range(ROT)]
    t_md = time_rotating([lambda o=o, yo=yo: ops.nvfp4_mxfp8_dequantize(o["q"], o["sf"], M, K, yo, K, stream)
                          for o, yo in zip(mx_out, ymx)])
    mq_bytes = M * K * 2 + 2 * (M * K + M * K / 32)     # read X once; both copies written
    md_bytes = M * K + M * K / 32 + M * K * 2
    result["mxfp8"] = {"quantize_row_col_ms": round(t_mq, 5),
                       "quantize_gbs": round(mq_bytes / (t_mq * 1e-3) / 1e9, 1),
                       "dequantize_ms": round(t_md, 5),
                       "dequantize_gbs": round(md_bytes / (t_md * 1e-3) / 1e9, 1),
                       "shape": [M, K], "timing": rot_note}
    result["gpu_launches"] += 3 * ROT * args.steps
    # NVFP4 backward GEMMs on the same layer (column-wise copies, one scale each):
    # dgrad dX = dY W and wgrad dW = dY^T X; dY is a synthetic gradient [M, N]
    dy = to_dev(W.small_matrix(77, M, N, std=1e-3))
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
    gbw = capture_graphs(torch, bw, stream)
    bw_ms = [[], []]
    for _ in range(args.steps):
        for i, g in enumerate(gbw):
            flush.zero_()
            e0, e1 = ev(), ev()
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            bw_ms[i].append(e0.elapsed_time(e1))
    t_dg, t_wg = float(np.mean(bw_ms[0])), float(np.mean(bw_ms[1]))
    result["backward"] = {"dgrad_ms": round(t_dg, 5), "wgrad_ms": round(t_wg, 5),
                          "dgrad_tflops": round(flop / (t_dg * 1e-3) / 1e12, 1),
                          "wgrad_tflops": round(flop / (t_wg * 1e-3) / 1e12, 1),
                          "shapes": {"dgrad": [M, K, N], "wgrad": [N, K, M]}}
    result["gpu_launches"] += 2 * args.steps
    if not args.no_moe:
        result["moe"] = run_moe(args, ops, W, torch, dev, stream, flush, world, fp4_peak, hbm_gbs)
        result["gpu_launches"] += result["moe"].pop("launches")
    st = ops.nvfp4_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status after the run: {ops.STATUS_NAMES.get(st)}")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl)
    if world > 1:
        torch.distributed.destroy_process_group()
    return result


def run_moe(args, ops, W, torch, dev, stream, flush, world, fp4_peak, hbm_gbs):
    """The MoE expert step of the Qwen3-30B-A3B workload at 4096 tokens, with
    expert weights quantized once (they are fixed within a step)."""
    wl = W.config3()
    m = wl.moe
    T, H, F, E, k = m.tokens, m.hidden, m.ffn, m.experts, m.topk

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    x = to_dev(m.x)
    ids = torch.from_numpy(m.topk_ids).to(dev)
    w1 = ops.quantize_experts(to_dev(m.w1))
    w2 = ops.quantize_experts(to_dev(m.w2))
    align = args.moe_row_align
    cap = ops.nvfp4_moe_capacity(T, k, E, align)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    gather = torch.empty(cap, dtype=torch.int32, device=dev)
    dst = torch.empty((T, k), dtype=torch.int32, device=dev)
    pws_b = ops.nvfp4_moe_permute_workspace_bytes(T, k, E)
    pws = torch.empty(pws_b, dtype=torch.uint8, device=dev)
    xq = dict(q=torch.empty((T, H // 2), dtype=torch.uint8, device=dev),
              sf=torch.empty(ops.nvfp4_sf_bytes(T, H), dtype=torch.uint8, device=dev),
              s=torch.empty(T, dtype=torch.float32, device=dev))
    a = dict(rows=cap, cols=H, q=torch.empty((cap, H // 2), dtype=torch.uint8, device=dev),
             sf=torch.empty(ops.nvfp4_sf_bytes(cap, H), dtype=torch.uint8, device=dev),
             s=torch.empty(cap, dtype=torch.float32, device=dev))
    y1 = torch.empty((cap, 2 * F), dtype=torch.bfloat16, device=dev)
    hq = dict(rows=cap, cols=F, q=torch.empty((cap, F // 2), dtype=torch.uint8, device=dev),
              sf=torch.empty(ops.nvfp4_sf_bytes(cap, F), dtype=torch.uint8, device=dev),
              s=torch.empty(cap, dtype=torch.float32, device=dev))
    y2 = torch.empty((cap, H), dtype=torch.bfloat16, device=dev)
    cw = torch.from_numpy(W.topk_weights(2, T, k)).to(dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    stages = [
        lambda: ops.nvfp4_moe_permute(ids, T, k, E, align, off, gather, cap, dst, pws, pws_b, stream),
        # per-token quantization of the tokens once, then their rows copied to the
        # routed layout (equal, bit for bit, to quantizing the gathered rows)
        lambda: ops.nvfp4_quantize_per_token(x, T, H, H, None, T, ops.PER_TOKEN, xq["q"], xq["sf"], xq["s"],
                                             stream=stream),
        lambda: ops.nvfp4_moe_gather_quantized(xq["q"], xq["sf"], xq["s"], T, H, gather, cap, a["q"], a["sf"],
                                               a["s"], stream),
        lambda: ops.nvfp4_grouped_gemm(a["q"], a["sf"], a["s"], cap, off, E, w1["q"], w1["sf"],
                                       w1["s"], 2 * F, H, y1, stream),
        lambda: ops.nvfp4_swiglu_quantize(y1, cap, F, 2 * F, off[E:], hq["q"], hq["sf"], hq["s"], None,
                                          stream),
        lambda: ops.nvfp4_grouped_gemm(hq["q"], hq["sf"], hq["s"], cap, off, E, w2["q"], w2["sf"],
                                       w2["s"], H, F, y2, stream),
        lambda: ops.nvfp4_moe_combine(y2, cap, H, dst, cw, T, k, H, out, H, stream),
    ]
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        for fn in stages:
            fn()
    torch.cuda.synchronize()
    graphs = capture_graphs(torch, stages, stream)

    def step(evs=None):
        for i, g in enumerate(graphs):
            if evs:
                evs[i].record(stream)
            g.replay()
        if evs:
            evs[len(graphs)].record(stream)

    runs = []
    for _ in range(args.steps):
        flush.zero_()
        evs = [ev() for _ in range(len(stages) + 1)]
        step(evs)
        runs.append(evs)
    torch.cuda.synchronize()
    ns = len(stages)
    seg = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(ns)] for e in runs]).mean(axis=0)
    # the whole step as one graph (the figure reported); the stage graphs above give the split
    (g_all,) = capture_graphs(torch, [lambda: [fn() for fn in stages]], stream)
    tot = []
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        g_all.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        tot.append(e0.elapsed_time(e1))
    total = float(np.mean(tot))
    routed = T * k
    flop = 2.0 * routed * H * 2 * F + 2.0 * routed * F * H
    fc1_flop = 2.0 * routed * H * 2 * F
    fc2_flop = 2.0 * routed * F * H
    used_rows = int(off[E].item())
    # weight bytes each grouped GEMM must read at least once (codes + scales + row scales)
    w1_bytes = E * (2 * F) * (H // 2 + H // 16 + 4)
    w2_bytes = E * H * (F // 2 + F // 16 + 4)
    # every byte a grouped GEMM must move at least once: its quantized input
    # rows (the padded layout's used rows), the expert weights and its bf16 output
    fc1_io = used_rows * (H // 2 + H // 16 + 4) + w1_bytes + used_rows * 2 * F * 2
    fc2_io = used_rows * (F // 2 + F // 16 + 4) + w2_bytes + used_rows * H * 2
    # SwiGLU-quantize: reads the used rows of Y1, writes codes, scales and S of
    # every row of the capacity (rows past the used ones are written as zeros)
    swi_io = used_rows * 2 * F * 2 + cap * (F // 2 + 4) + ops.nvfp4_sf_bytes(cap, F)

    def gbs(nbytes, ms):
        return round(nbytes / (ms * 1e-3) / 1e9, 1)
    return {
        "workload": "qwen3_30b_a3b_moe_4096tok_128e_top8 (hidden 2048, expert ffn 768)",
        "ms_per_step": round(total, 5),
        "stage_graphs_ms": round(float(np.array([e[0].elapsed_time(e[ns]) for e in runs]).mean()), 5),
        "launch": "the step captured as one CUDA graph; kernels_ms from one graph per stage",
        "tflops": round(world * flop / (total * 1e-3) / 1e12, 2),
        "padded_rows": used_rows, "routed_rows": routed, "row_align": align,
        "kernels_ms": {"permute": round(seg[0], 5), "quantize_tokens": round(seg[1], 5),
                       "gather_quantized": round(seg[2], 5), "grouped_fc1": round(seg[3], 5),
                       "swiglu_quantize": round(seg[4], 5), "grouped_fc2": round(seg[5], 5),
                       "combine": round(seg[6], 5)},
        # combine: reads top-k rows of the fc2 output per token, writes one row
        "combine_gbs": round((routed * H * 2 + T * H * 2 + routed * 8) / (seg[6] * 1e-3) / 1e9, 1),
        "grouped_fc1": {"tflops": round(fc1_flop / (seg[3] * 1e-3) / 1e12, 1),
                        "frac_of_fp4_peak": round(fc1_flop / (seg[3] * 1e-3) / 1e12 / fp4_peak, 4),
                        "weight_gbs": gbs(w1_bytes, seg[3]),
                        "weight_frac_of_hbm": round(gbs(w1_bytes, seg[3]) / hbm_gbs, 4),
                        "io_bytes": int(fc1_io), "io_gbs": gbs(fc1_io, seg[3]),
                        "io_frac_of_hbm": round(gbs(fc1_io, seg[3]) / hbm_gbs, 4)},
        "grouped_fc2": {"tflops": round(fc2_flop / (seg[5] * 1e-3) / 1e12, 1),
                        "frac_of_fp4_peak": round(fc2_flop / (seg[5] * 1e-3) / 1e12 / fp4_peak, 4),
                        "weight_gbs": gbs(w2_bytes, seg[5]),
                        "weight_frac_of_hbm": round(gbs(w2_bytes, seg[5]) / hbm_gbs, 4),
                        "io_bytes": int(fc2_io), "io_gbs": gbs(fc2_io, seg[5]),
                        "io_frac_of_hbm": round(gbs(fc2_io, seg[5]) / hbm_gbs, 4)},
        "swiglu_quantize": {"io_bytes": int(swi_io), "io_gbs": gbs(swi_io, seg[4]),
                            "io_frac_of_hbm": round(gbs(swi_io, seg[4]) / hbm_gbs, 4)},
        "launches": 18 * args.steps,   # stage graphs + one-graph step, 9 kernels each
    }


# ----------------------------------------------------------------------------
# CPU oracle timings (baseline and the reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(wl, rows_x, rows_w, nthreads):
    """One bounded sample of the step on the oracle: quantize rows_x rows of X
    and rows_w rows of W, then their exact W4A4 product.  Returns (flop, s)."""
    import oracle
    t0 = time.perf_counter()
    a = oracle.quantize(wl.x[:rows_x], nthreads=nthreads)
    b = oracle.quantize(wl.w[:rows_w], nthreads=nthreads)
    oracle.gemm_exact(a, b, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return 2.0 * rows_x * rows_w * K, dt


def cpu_baseline(wl, target_s=12.0):
    import oracle
    cores = os.cpu_count() or 1
    rx, rw = 128, 1024
    flop, dt = oracle_sample(wl, rx, rw, cores)
    reps = max(1, int(target_s / max(dt, 1e-3)))
    tot_f, tot_t = 0.0, 0.0
    for _ in range(min(reps, 200)):
        f, t = oracle_sample(wl, rx, rw, cores)
        tot_f += f
        tot_t += t
    return {"value": round(tot_f / tot_t / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"quantize {rx} rows of X and {rw} rows of W (per-token), exact int64 W4A4 "
                      f"product {rx}x{rw}x{K}; {min(reps, 200)} repetitions, {tot_t:.1f} s"}


def run_reference(args):
    from nvfp4_precision_rl_gb300 import workloads as W
    wl = W.config2()
    cores = os.cpu_count() or 1
    rx, rw = 128, 1024
    for _ in range(args.warmup):
        oracle_sample(wl, rx, rw, cores)
    flops, times = 0.0, []
    for _ in range(args.steps):
        f, t = oracle_sample(wl, rx, rw, cores)
        flops = f
        times.append(t)
    ms = float(np.mean(times)) * 1e3
    value = flops / (ms * 1e-3) / 1e12
    sample = (f"per step: quantize {rx} rows of X and {rw} rows of W (per-token), exact int64 "
              f"W4A4 product {rx}x{rw}x{K} on {cores} host threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64 exact / f64",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": WORKLOAD, "M_tokens": M, "N": N, "K": K, "seq_len": 4096,
                   "micro_batch": 1, "sample_rows_x": rx, "sample_rows_w": rw},
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
