"""CPU oracle for the per-token NVFP4 W4A4 linear-layer path.

TEST INFRASTRUCTURE ONLY: only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference arm may import this package.  The product library
(nvfp4_precision_rl_gb300) never imports it, and it never imports the product
library; the two share only the seeded input generators, which hold none of the
method's arithmetic.

All arithmetic lives in nvfp4_oracle.c (plain C, one IEEE binary32 operation
per step of the quantizer, exact integer GEMM); this module only marshals numpy
arrays through ctypes.  Every function cites the passage it follows there.

Parity status per function (what pins it is in tests/test_oracle_*.py):
  e2m1/e4m3 tables and encoders  pinned (value set printed on the pages,
                                 torch float8_e4m3fn, banker's-rounding form)
  quantize_rows / quantize_cols  pinned (round trip, error bound, batch
                                 invariance, zeros / maxes / boundary classes)
  sf_swizzle                     pinned (bijection + hand-derived positions;
                                 the GPU GEMM consumes it)
  gemm_exact / gemm_fp64         pinned (brute force, integer special case,
                                 float64 matmul of the decoded operands)
  moe_permute                    pinned (numpy stable argsort, invariants)
  swiglu                         pinned (float64 closed form on exact inputs)
  dequantize_bf16                pinned (hand-worked values, exact binary64
                                 product within one bf16 rounding, round trip)
  mxfp8_quantize / dequantize    pinned (hand-worked blocks, the rounded-up
                                 scale's minimality, torch float8_e4m3fn
                                 codec, exact dequantization, round trip)
  moe_combine                    pinned (top-1 unit weight = the inverse
                                 permutation; exact dyadic sums; binary64 sum
                                 within the binary32 bound; slot order)
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        L.orc_e2m1_table.argtypes = [P]
        L.orc_e4m3_table.argtypes = [P]
        L.orc_e2m1_encode.argtypes = [P, I64, P]
        L.orc_e4m3_encode.argtypes = [P, I64, P]
        L.orc_quantize_rows.argtypes = [P, I64, I64, P, I64, ctypes.c_int, P, P, P, ctypes.c_int]
        L.orc_quantize_rows.restype = ctypes.c_float
        L.orc_quantize_cols.argtypes = [P, I64, I64, P, I64, ctypes.c_float, P, P, ctypes.c_int]
        L.orc_quantize_cols.restype = ctypes.c_float
        L.orc_sf_swizzled_bytes.argtypes = [I64, I64]
        L.orc_sf_swizzled_bytes.restype = I64
        L.orc_sf_swizzle.argtypes = [P, I64, I64, P]
        L.orc_sf_unswizzle.argtypes = [P, I64, I64, P]
        L.orc_dequantize.argtypes = [P, P, P, I64, I64, P]
        L.orc_gemm_exact.argtypes = [P, P, P, I64, P, P, P, I64, I64, P, P, ctypes.c_int]
        L.orc_gemm_exact_sampled.argtypes = [P, P, P, I64, P, P, P, I64, I64, P, P, I64, P, P,
                                             ctypes.c_int]
        L.orc_gemm_fp64.argtypes = [P, P, P, I64, P, P, P, I64, I64, P]
        L.orc_moe_permute.argtypes = [P, I64, I32, I32, I32, P, P, I64, P]
        L.orc_moe_permute.restype = ctypes.c_int
        L.orc_swiglu.argtypes = [P, I64, I64, I64, P]
        L.orc_bf16_from_double.argtypes = [P, I64, P]
        L.orc_dequantize_bf16.argtypes = [P, P, P, ctypes.c_int, I64, I64, P]
        L.orc_moe_combine.argtypes = [P, I64, I64, P, P, I64, ctypes.c_int, I64, P]
        L.orc_mxfp8_quantize_rows.argtypes = [P, I64, I64, I64, P, P]
        L.orc_mxfp8_quantize_cols.argtypes = [P, I64, I64, I64, P, P]
        L.orc_mxfp8_dequantize_bf16.argtypes = [P, P, I64, I64, P]
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads():
    return os.cpu_count() or 1


# -- formats ------------------------------------------------------------------

def e2m1_table():
    out = np.zeros(16, np.float64)
    lib().orc_e2m1_table(_p(out))
    return out


def e4m3_table():
    out = np.zeros(256, np.float64)
    lib().orc_e4m3_table(_p(out))
    return out


def e2m1_encode(x):
    x = _c(x, np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    lib().orc_e2m1_encode(_p(x), x.size, _p(out))
    return out


def e4m3_encode(x):
    x = _c(x, np.float32).ravel()
    out = np.zeros(x.size, np.uint8)
    lib().orc_e4m3_encode(_p(x), x.size, _p(out))
    return out


# -- quantizer -------------------------------------------------------------------

def sf_swizzled_bytes(rows, kb):
    return int(lib().orc_sf_swizzled_bytes(rows, kb))


def sf_swizzle(sf_rm):
    sf_rm = _c(sf_rm, np.uint8)
    rows, kb = sf_rm.shape
    out = np.zeros(sf_swizzled_bytes(rows, kb), np.uint8)
    lib().orc_sf_swizzle(_p(sf_rm), rows, kb, _p(out))
    return out


def sf_unswizzle(swz, rows, kb):
    swz = _c(swz, np.uint8)
    out = np.zeros((rows, kb), np.uint8)
    lib().orc_sf_unswizzle(_p(swz), rows, kb, _p(out))
    return out


def quantize(x_bf16, gather=None, rows_out=None, mode="per_token", column_copy=False,
             nthreads=None):
    """Two-level NVFP4 quantization of the rows of a bf16 matrix (uint16 bits).

    Returns a dict with q [rows_out, cols/2] uint8, sf [rows_out, cols/16] E4M3
    codes (row-major), sf_swz (the swizzled layout), s [rows_out] float32, amax,
    and with column_copy the X^T copy: q_col, sf_col, sf_col_swz, s_col.
    """
    x = _c(x_bf16, np.uint16)
    rows_in, cols = x.shape
    if gather is not None:
        gather = _c(gather, np.int32)
        rows_out = gather.size if rows_out is None else rows_out
        assert gather.size >= rows_out
    else:
        rows_out = rows_in if rows_out is None else rows_out
        assert rows_out <= rows_in
    assert cols % 16 == 0
    nt = default_threads() if nthreads is None else nthreads
    q = np.zeros((rows_out, cols // 2), np.uint8)
    sf = np.zeros((rows_out, cols // 16), np.uint8)
    s = np.zeros(rows_out, np.float32)
    amax = lib().orc_quantize_rows(_p(x), cols, cols, _p(gather), rows_out,
                                   1 if mode == "per_tensor" else 0, _p(q), _p(sf), _p(s), nt)
    out = dict(q=q, sf=sf, s=s, amax=np.float32(amax), sf_swz=sf_swizzle(sf))
    if column_copy:
        assert rows_out % 16 == 0
        qc = np.zeros((cols, rows_out // 2), np.uint8)
        sfc = np.zeros((cols, rows_out // 16), np.uint8)
        s_col = lib().orc_quantize_cols(_p(x), cols, cols, _p(gather), rows_out,
                                        ctypes.c_float(amax), _p(qc), _p(sfc), nt)
        out.update(q_col=qc, sf_col=sfc, sf_col_swz=sf_swizzle(sfc),
                   s_col=np.array([s_col], np.float32))
    return out


def dequantize(q, sf_rm, s):
    q = _c(q, np.uint8)
    sf_rm = _c(sf_rm, np.uint8)
    s = _c(s, np.float32)
    rows = q.shape[0]
    cols = q.shape[1] * 2
    out = np.zeros((rows, cols), np.float64)
    lib().orc_dequantize(_p(q), _p(sf_rm), _p(s), rows, cols, _p(out))
    return out


def dequantize_bf16(q, sf_rm, s, s_per_row=True):
    """bf16 bits of y = bf16_rn(fl32(S * dec(q) * dec(s_b))) (row-major scales)."""
    q = _c(q, np.uint8)
    sf_rm = _c(sf_rm, np.uint8)
    s = _c(s, np.float32)
    rows = q.shape[0]
    cols = q.shape[1] * 2
    out = np.zeros((rows, cols), np.uint16)
    lib().orc_dequantize_bf16(_p(q), _p(sf_rm), _p(s), 1 if s_per_row else 0, rows, cols, _p(out))
    return out


# -- GEMM ----------------------------------------------------------------------

def gemm_exact(a, b, with_abs=False, nthreads=None):
    """Y[m, n] = sum_k x^[m,k] w^[n,k] from two quantize() results (exact int64)."""
    qa, sfa, sa = _c(a["q"], np.uint8), _c(a["sf"], np.uint8), _c(a["s"], np.float32)
    qb, sfb, sb = _c(b["q"], np.uint8), _c(b["sf"], np.uint8), _c(b["s"], np.float32)
    M, K = qa.shape[0], qa.shape[1] * 2
    N = qb.shape[0]
    assert qb.shape[1] * 2 == K
    y = np.zeros((M, N), np.float64)
    absy = np.zeros((M, N), np.float64) if with_abs else None
    nt = default_threads() if nthreads is None else nthreads
    lib().orc_gemm_exact(_p(qa), _p(sfa), _p(sa), M, _p(qb), _p(sfb), _p(sb), N, K, _p(y),
                         _p(absy), nt)
    return (y, absy) if with_abs else y


def gemm_exact_sampled(a, b, mi, ni, nthreads=None):
    """Exact Y at the listed (mi[i], ni[i]); returns (y, sum of |products|)."""
    qa, sfa, sa = _c(a["q"], np.uint8), _c(a["sf"], np.uint8), _c(a["s"], np.float32)
    qb, sfb, sb = _c(b["q"], np.uint8), _c(b["sf"], np.uint8), _c(b["s"], np.float32)
    M, K = qa.shape[0], qa.shape[1] * 2
    N = qb.shape[0]
    mi = _c(mi, np.int64)
    ni = _c(ni, np.int64)
    y = np.zeros(mi.size, np.float64)
    absy = np.zeros(mi.size, np.float64)
    nt = default_threads() if nthreads is None else nthreads
    lib().orc_gemm_exact_sampled(_p(qa), _p(sfa), _p(sa), M, _p(qb), _p(sfb), _p(sb), N, K,
                                 _p(mi), _p(ni), mi.size, _p(y), _p(absy), nt)
    return y, absy


def gemm_fp64(a, b):
    qa, sfa, sa = _c(a["q"], np.uint8), _c(a["sf"], np.uint8), _c(a["s"], np.float32)
    qb, sfb, sb = _c(b["q"], np.uint8), _c(b["sf"], np.uint8), _c(b["s"], np.float32)
    M, K = qa.shape[0], qa.shape[1] * 2
    N = qb.shape[0]
    y = np.zeros((M, N), np.float64)
    lib().orc_gemm_fp64(_p(qa), _p(sfa), _p(sa), M, _p(qb), _p(sfb), _p(sb), N, K, _p(y))
    return y


def rows_of(d, r0, r1):
    """Rows [r0, r1) of a quantize() result, as an operand for the GEMM."""
    return dict(q=d["q"][r0:r1], sf=d["sf"][r0:r1], s=d["s"][r0:r1])


# -- MoE -----------------------------------------------------------------------

def moe_capacity(tokens, topk, num_experts, align):
    """Rows the padded per-expert layout can need at most."""
    return tokens * topk + num_experts * (align - 1)


def moe_permute(topk_ids, num_experts, align=128, capacity=None):
    topk_ids = _c(topk_ids, np.int32)
    T, k = topk_ids.shape
    cap = moe_capacity(T, k, num_experts, align) if capacity is None else capacity
    offsets = np.zeros(num_experts + 1, np.int32)
    gather = np.zeros(cap, np.int32)
    dst = np.zeros(T * k, np.int32)
    rc = lib().orc_moe_permute(_p(topk_ids), T, k, num_experts, align, _p(offsets), _p(gather),
                               cap, _p(dst))
    if rc != 0:
        raise ValueError("moe_permute: expert id out of range or capacity too small")
    return dict(offsets=offsets, gather=gather, dst=dst.reshape(T, k), capacity=cap)


def mxfp8_quantize(x_bf16, column_copy=False):
    """MXFP8 of bf16 [rows, cols]: q [rows, cols] E4M3 codes, sf [rows, cols/32]
    E8M0 codes (row-major) and sf_swz (the 128 x 4 tile layout); with
    column_copy the 32x1 copy of X^T: q_col [cols, rows], sf_col, sf_col_swz."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    q = np.zeros((rows, cols), np.uint8)
    sf = np.zeros((rows, cols // 32), np.uint8)
    lib().orc_mxfp8_quantize_rows(_p(x), rows, cols, cols, _p(q), _p(sf))
    out = dict(q=q, sf=sf, sf_swz=sf_swizzle(sf))
    if column_copy:
        qc = np.zeros((cols, rows), np.uint8)
        sfc = np.zeros((cols, rows // 32), np.uint8)
        lib().orc_mxfp8_quantize_cols(_p(x), rows, cols, cols, _p(qc), _p(sfc))
        out.update(q_col=qc, sf_col=sfc, sf_col_swz=sf_swizzle(sfc))
    return out


def mxfp8_dequantize_bf16(q, sf_rm):
    q = _c(q, np.uint8)
    sf_rm = _c(sf_rm, np.uint8)
    rows, cols = q.shape
    out = np.zeros((rows, cols), np.uint16)
    lib().orc_mxfp8_dequantize_bf16(_p(q), _p(sf_rm), rows, cols, _p(out))
    return out


def moe_combine(y2_bf16, dst_rows, weights):
    """out[t] = bf16(sum_j w[t, j] * y2[dst[t, j]]) in binary32, slot order."""
    y2 = _c(y2_bf16, np.uint16)
    dst = _c(dst_rows, np.int32).ravel()
    w = _c(weights, np.float32)
    tokens, topk = w.shape
    assert dst.size == tokens * topk
    rows, hidden = y2.shape
    out = np.zeros((tokens, hidden), np.uint16)
    lib().orc_moe_combine(_p(y2), rows, hidden, _p(dst), _p(w), tokens, topk, hidden, _p(out))
    return out


def swiglu(y1_bf16, F):
    y1 = _c(y1_bf16, np.uint16)
    rows = y1.shape[0]
    h = np.zeros((rows, F), np.uint16)
    lib().orc_swiglu(_p(y1), rows, F, y1.shape[1], _p(h))
    return h


def bf16_from_double(v):
    v = _c(v, np.float64).ravel()
    out = np.zeros(v.size, np.uint16)
    lib().orc_bf16_from_double(_p(v), v.size, _p(out))
    return out
