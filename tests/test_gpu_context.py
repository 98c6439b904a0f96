"""The library's cached device addresses (the status word, the no-alloc
permute's scratch array) and per-kernel attributes belong to one CUDA context.
With a second context made current on the same device, every call must look
them up again in that context, and switching back must find the first
context's again: the same calls in both contexts give the same bytes, with the
device status OK, and the first context's bytes match the oracle.

Runs in a child process that drives the CUDA driver API directly (its own
contexts and buffers, no torch), so the contexts it creates and destroys never
touch the test session's.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import ctypes, sys
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    from nvfp4_precision_rl_gb300 import ops, workloads as W

    cu = ctypes.CDLL("libcuda.so.1")
    def ck(r, what):
        if r != 0:
            raise RuntimeError(f"{what}: CUresult {r}")
    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int()
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "retain")
    ck(cu.cuCtxSetCurrent(primary), "set primary")
    L = ops.lib()

    M = N = 256
    K = 512
    T, k, E = 4096, 8, 128
    x = W.small_matrix(71, M, K)
    w = W.small_matrix(72, N, K, std=0.02)
    ids = W.route_topk(np.random.default_rng(73), T, E, k)
    cap = int(L.nvfp4_moe_capacity(T, k, E, 128))
    sfb = int(L.nvfp4_sf_bytes(M, K))

    def run():
        # buffers of the current context, the calls, the bytes back
        bufs = []
        def alloc(nbytes, host=None):
            p = ctypes.c_uint64()
            ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "alloc")
            bufs.append(p.value)
            if host is not None:
                h = np.ascontiguousarray(host)
                ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p.value), h.ctypes.data_as(ctypes.c_void_p),
                                      ctypes.c_size_t(h.nbytes)), "h2d")
            return p.value
        def back(ptr, shape, dtype):
            h = np.empty(shape, dtype)
            ck(cu.cuCtxSynchronize(), "sync")
            ck(cu.cuMemcpyDtoH_v2(h.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(ptr),
                                  ctypes.c_size_t(h.nbytes)), "d2h")
            return h
        dx, dw = alloc(x.nbytes, x), alloc(w.nbytes, w)
        qx, sfx, sx = alloc(M * K // 2), alloc(sfb), alloc(M * 4)
        qw, sfw, sw = alloc(N * K // 2), alloc(sfb), alloc(N * 4)
        y = alloc(M * N * 2)
        dids = alloc(ids.nbytes, ids)
        off, gat, dst = alloc((E + 1) * 4), alloc(cap * 4), alloc(T * k * 4)
        for src, q, sf, s, rows in ((dx, qx, sfx, sx, M), (dw, qw, sfw, sw, N)):
            assert L.nvfp4_quantize_per_token(src, rows, K, K, None, rows, 0, q, sf, s, None, None, None,
                                              None, 0, None) == 0
        assert L.nvfp4_gemm(qx, sfx, sx, M, qw, sfw, sw, N, K, y, N, None) == 0
        for _ in range(2):
            assert L.nvfp4_moe_permute_noalloc(dids, T, k, E, 128, off, gat, cap, dst, None) == 0
        out = dict(q=back(qx, (M, K // 2), np.uint8), sf=back(sfx, sfb, np.uint8), s=back(sx, M, np.float32),
                   y=back(y, (M, N), np.uint16), off=back(off, E + 1, np.int32), gather=back(gat, cap, np.int32),
                   dst=back(dst, (T, k), np.int32))
        assert L.nvfp4_get_device_status(None) == 0, "device status"
        for p in bufs:
            ck(cu.cuMemFree_v2(ctypes.c_uint64(p)), "free")
        return out

    a = run()
    rq = oracle.quantize(x)
    assert np.array_equal(a["q"], rq["q"]) and np.array_equal(a["sf"], rq["sf_swz"])
    assert np.array_equal(a["s"].view(np.uint32), rq["s"].view(np.uint32))
    rp = oracle.moe_permute(ids, E, 128, capacity=cap)
    assert np.array_equal(a["off"], rp["offsets"]) and np.array_equal(a["gather"], rp["gather"])
    assert np.array_equal(a["dst"], rp["dst"])

    second = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(second), 0, dev), "create")   # current from here on
    b = run()
    ck(cu.cuCtxSetCurrent(primary), "back to primary")
    c = run()
    ck(cu.cuCtxDestroy_v2(second), "destroy")
    for key in a:
        assert np.array_equal(a[key], b[key]), f"{key} differs in the second context"
        assert np.array_equal(a[key], c[key]), f"{key} differs back in the first context"
    ck(cu.cuDevicePrimaryCtxRelease_v2(dev), "release")
    print("CONTEXTS_OK")
""")


def test_calls_follow_the_current_context(nv):
    code = f"ROOT = {ROOT!r}\n" + CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "CONTEXTS_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
