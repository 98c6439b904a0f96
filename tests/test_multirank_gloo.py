"""The N > 1 path on CPU with the gloo backend (world size 2, 127.0.0.1).

bench.py shards the work by rows across ranks with no data-path collective:
each rank runs its own batch, and only the step time is reduced (max over
ranks).  Per-token scales make that sharding exact: a rank's quantized rows are
byte-identical to the same rows quantized in the unsharded matrix (checked here
with the oracle on CPU), so no amax exchange is needed.  Only a per-tensor
scale would need one (an all-reduce of the amax), which the test also shows.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from nvfp4_precision_rl_gb300 import workloads as W
        # timing reduction: the job's step time is the slowest rank's
        t = bench.max_over_ranks(1.0 + rank, "cpu", world)
        thr = bench.job_throughput(100.0, world, t)
        # row-sharded per-token quantization equals the unsharded result
        x = W.small_matrix(5, 96, 256, dist="student_t3", outlier_cols=4, outlier_scale=50)
        rows = np.array_split(np.arange(96), world)[rank]
        mine = oracle.quantize(x[rows], nthreads=1)
        full = oracle.quantize(x, nthreads=1)
        same = bool(np.array_equal(mine["q"], full["q"][rows]) and
                    np.array_equal(mine["s"], full["s"][rows]))
        # a per-tensor scale is not shard-local: it needs the global amax
        local_amax = torch.tensor([float(mine["amax"])])
        dist.all_reduce(local_amax, op=dist.ReduceOp.MAX)
        pt_local = oracle.quantize(x[rows], mode="per_tensor", nthreads=1)
        pt_full = oracle.quantize(x, mode="per_tensor", nthreads=1)
        q.put((rank, t, thr, same, float(local_amax.item()) == float(full["amax"]),
               bool(np.array_equal(pt_local["q"], pt_full["q"][rows]))))
    finally:
        dist.destroy_process_group()


def test_two_rank_reduction_and_sharding():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=240) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, thr, same, amax_ok, pt_same in results:
        assert t == 2.0                      # max over ranks of (1.0 + rank)
        assert thr == pytest.approx(100.0 * world / 2.0)
        assert same                          # per-token: shard bytes == unsharded bytes
        assert amax_ok                       # the all-reduced amax is the tensor's
    assert not all(r[5] for r in results)    # per-tensor: at least one shard differs
