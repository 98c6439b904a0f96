"""Thin Python binding of libnvfp4 (include/nvfp4.h): argument marshalling only.

Every function named nvfp4_* calls the C entry point of the same name with raw
device pointers taken from torch tensors and the current CUDA stream; every
step of the computation runs in the library's CUDA kernels.  The lower-case
helpers (quantize, gemm, ...) only allocate the output tensors with torch and
call those entry points.  If the library is not built the import of a helper
fails loudly: there is no CPU or PyTorch fallback.
"""
import ctypes
import os

import torch

from . import _build

_LIB = None

STATUS_NAMES = {
    0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_ALIGNMENT", 3: "NVFP4_ERR_SHAPE",
    4: "NVFP4_ERR_UNSUPPORTED_DEVICE", 5: "NVFP4_ERR_CUDA", 6: "NVFP4_ERR_TIMEOUT",
    7: "NVFP4_ERR_DEVICE_INPUT", 8: "NVFP4_ERR_WORKSPACE",
}
PER_TOKEN, PER_TENSOR = 0, 1


class NVFP4Error(RuntimeError):
    def __init__(self, where, status):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")
        self.status = status


def library_path():
    return _build.LIB


def lib():
    """Load libnvfp4.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libnvfp4.so is not built (expected {path}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    st = ctypes.c_int
    sig = {
        "nvfp4_packed_bytes": (SZ, [I64, I64]),
        "nvfp4_sf_bytes": (SZ, [I64, I64]),
        "nvfp4_quantize_workspace_bytes": (SZ, []),
        "nvfp4_quantize_per_token": (st, [P, I64, I64, I64, P, I64, ctypes.c_int, P, P, P, P, P, P,
                                          P, SZ, P]),
        "nvfp4_moe_capacity": (I64, [I64, I32, I32, I32]),
        "nvfp4_moe_permute_workspace_bytes": (SZ, [I64, I32, I32]),
        "nvfp4_moe_permute": (st, [P, I64, I32, I32, I32, P, P, I64, P, P, SZ, P]),
        "nvfp4_moe_permute_noalloc": (st, [P, I64, I32, I32, I32, P, P, I64, P, P]),
        "nvfp4_gemm": (st, [P, P, P, I64, P, P, P, I64, I64, P, I64, P]),
        "nvfp4_grouped_gemm": (st, [P, P, P, I64, P, I32, P, P, P, I64, I64, P, P]),
        "nvfp4_grouped_gemm_swiglu": (st, [P, P, P, I64, P, I32, P, P, P, I64, I64, P, P]),
        "nvfp4_swiglu_quantize": (st, [P, I64, I64, I64, P, P, P, P, P, P]),
        "nvfp4_dequantize": (st, [P, P, P, ctypes.c_int32, I64, I64, P, I64, P]),
        "nvfp4_gemm_ex": (st, [P, P, P, ctypes.c_int32, I64, P, P, P, ctypes.c_int32, I64, I64, P, I64, P]),
        "nvfp4_quantize_per_token_pair": (st, [P, I64, I64, P, P, P, P, P, P, P, I64, I64, P, P, P, I64, P,
                                               SZ, P]),
        "nvfp4_moe_combine": (st, [P, I64, I64, P, P, I64, ctypes.c_int32, I64, P, I64, P]),
        "nvfp4_moe_gather_quantized": (st, [P, P, P, I64, I64, P, I64, P, I32, P, P, P, P]),
        "nvfp4_mxfp8_sf_bytes": (SZ, [I64, I64]),
        "nvfp4_mxfp8_quantize": (st, [P, I64, I64, I64, P, P, P, P, P]),
        "nvfp4_mxfp8_dequantize": (st, [P, P, I64, I64, P, I64, P]),
        "nvfp4_get_device_status": (st, [P]),
        "nvfp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "nvfp4_debug_cvt_probe": (st, [P, P, P, P]),
        "nvfp4_debug_scale_recipe_check": (st, [P, P, P]),
        "nvfp4_debug_wait_timeout": (st, [I64, P]),
        "nvfp4_debug_set_gemm_wait_limit": (st, [I64]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = L
    return L


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _ok(name, status):
    if status != 0:
        raise NVFP4Error(name, status)


# ---------------------------------------------------------------------------
# The C entry points, one to one
# ---------------------------------------------------------------------------

def nvfp4_packed_bytes(rows, cols):
    return lib().nvfp4_packed_bytes(rows, cols)


def nvfp4_sf_bytes(rows, cols):
    return lib().nvfp4_sf_bytes(rows, cols)


def nvfp4_quantize_workspace_bytes():
    return lib().nvfp4_quantize_workspace_bytes()


def nvfp4_quantize_per_token(x, rows_in, cols, ld_x, gather_rows, rows_out, mode, q_row, sf_row,
                             s_row, q_col=None, sf_col=None, s_col=None, workspace=None,
                             workspace_bytes=0, stream=None):
    _ok("nvfp4_quantize_per_token", lib().nvfp4_quantize_per_token(
        _p(x), rows_in, cols, ld_x, _p(gather_rows), rows_out, mode, _p(q_row), _p(sf_row),
        _p(s_row), _p(q_col), _p(sf_col), _p(s_col), _p(workspace), workspace_bytes, _s(stream)))


def nvfp4_moe_capacity(tokens, topk, num_experts, row_align):
    return lib().nvfp4_moe_capacity(tokens, topk, num_experts, row_align)


def nvfp4_moe_permute_workspace_bytes(tokens, topk, num_experts):
    return lib().nvfp4_moe_permute_workspace_bytes(tokens, topk, num_experts)


def nvfp4_moe_permute(topk_ids, tokens, topk, num_experts, row_align, expert_offsets, gather_rows,
                      capacity, dst_rows, workspace, workspace_bytes, stream=None):
    _ok("nvfp4_moe_permute", lib().nvfp4_moe_permute(
        _p(topk_ids), tokens, topk, num_experts, row_align, _p(expert_offsets), _p(gather_rows),
        capacity, _p(dst_rows), _p(workspace), workspace_bytes, _s(stream)))


def nvfp4_moe_permute_noalloc(topk_ids, tokens, topk, num_experts, row_align, expert_offsets,
                              gather_rows, capacity, dst_rows, stream=None):
    """nvfp4_moe_permute without a caller workspace (for callers that cannot
    allocate): the library's fixed 1 MiB scratch array is used instead."""
    _ok("nvfp4_moe_permute_noalloc", lib().nvfp4_moe_permute_noalloc(
        _p(topk_ids), tokens, topk, num_experts, row_align, _p(expert_offsets), _p(gather_rows),
        capacity, _p(dst_rows), _s(stream)))


def nvfp4_gemm(a_q, a_sf, a_s, M, b_q, b_sf, b_s, N, K, y, ld_y, stream=None):
    _ok("nvfp4_gemm", lib().nvfp4_gemm(_p(a_q), _p(a_sf), _p(a_s), M, _p(b_q), _p(b_sf), _p(b_s),
                                       N, K, _p(y), ld_y, _s(stream)))


def nvfp4_grouped_gemm(a_q, a_sf, a_s, rows_capacity, expert_offsets, E, b_q, b_sf, b_s, N, K, y,
                       stream=None):
    _ok("nvfp4_grouped_gemm", lib().nvfp4_grouped_gemm(
        _p(a_q), _p(a_sf), _p(a_s), rows_capacity, _p(expert_offsets), E, _p(b_q), _p(b_sf),
        _p(b_s), N, K, _p(y), _s(stream)))


def nvfp4_grouped_gemm_swiglu(a_q, a_sf, a_s, rows_capacity, expert_offsets, E, b_q, b_sf, b_s, ffn, K, h,
                              stream=None):
    _ok("nvfp4_grouped_gemm_swiglu", lib().nvfp4_grouped_gemm_swiglu(
        _p(a_q), _p(a_sf), _p(a_s), rows_capacity, _p(expert_offsets), E, _p(b_q), _p(b_sf), _p(b_s), ffn, K,
        _p(h), _s(stream)))


def nvfp4_moe_combine(y2, rows, ld_y2, dst_rows, weights, tokens, topk, hidden, out, ld_out, stream=None):
    _ok("nvfp4_moe_combine", lib().nvfp4_moe_combine(
        _p(y2), rows, ld_y2, _p(dst_rows), _p(weights), tokens, int(topk), hidden, _p(out), ld_out,
        _s(stream)))


def nvfp4_quantize_per_token_pair(x, rows_x, ld_x, q_x, sf_x, s_x, q_col, sf_col, s_col, w, rows_w, ld_w,
                                  q_w, sf_w, s_w, cols, workspace=None, workspace_bytes=0, stream=None):
    _ok("nvfp4_quantize_per_token_pair", lib().nvfp4_quantize_per_token_pair(
        _p(x), rows_x, ld_x, _p(q_x), _p(sf_x), _p(s_x), _p(q_col), _p(sf_col), _p(s_col), _p(w), rows_w, ld_w,
        _p(q_w), _p(sf_w), _p(s_w), cols, _p(workspace), workspace_bytes, _s(stream)))


def nvfp4_gemm_ex(a_q, a_sf, a_s, a_s_per_row, M, b_q, b_sf, b_s, b_s_per_row, N, K, y, ld_y, stream=None):
    _ok("nvfp4_gemm_ex", lib().nvfp4_gemm_ex(
        _p(a_q), _p(a_sf), _p(a_s), int(a_s_per_row), M, _p(b_q), _p(b_sf), _p(b_s), int(b_s_per_row), N, K,
        _p(y), ld_y, _s(stream)))


def nvfp4_dequantize(q, sf, s, s_per_row, rows, cols, y, ld_y, stream=None):
    _ok("nvfp4_dequantize", lib().nvfp4_dequantize(
        _p(q), _p(sf), _p(s), int(s_per_row), rows, cols, _p(y), ld_y, _s(stream)))


def nvfp4_moe_gather_quantized(q_src, sf_src, s_src, rows_src, cols, gather_rows, rows_out, expert_offsets,
                               num_experts, q, sf, s, stream=None):
    _ok("nvfp4_moe_gather_quantized", lib().nvfp4_moe_gather_quantized(
        _p(q_src), _p(sf_src), _p(s_src), rows_src, cols, _p(gather_rows), rows_out, _p(expert_offsets),
        num_experts, _p(q), _p(sf), _p(s), _s(stream)))


def nvfp4_mxfp8_sf_bytes(rows, cols):
    return int(lib().nvfp4_mxfp8_sf_bytes(rows, cols))


def nvfp4_mxfp8_quantize(x, rows, cols, ld_x, q, sf, q_col=None, sf_col=None, stream=None):
    _ok("nvfp4_mxfp8_quantize", lib().nvfp4_mxfp8_quantize(
        _p(x), rows, cols, ld_x, _p(q), _p(sf), _p(q_col), _p(sf_col), _s(stream)))


def nvfp4_mxfp8_dequantize(q, sf, rows, cols, y, ld_y, stream=None):
    _ok("nvfp4_mxfp8_dequantize", lib().nvfp4_mxfp8_dequantize(
        _p(q), _p(sf), rows, cols, _p(y), ld_y, _s(stream)))


def nvfp4_swiglu_quantize(y1, rows, ffn, ld_y1, row_count, q, sf, s, h=None, stream=None):
    _ok("nvfp4_swiglu_quantize", lib().nvfp4_swiglu_quantize(
        _p(y1), rows, ffn, ld_y1, _p(row_count), _p(q), _p(sf), _p(s), _p(h), _s(stream)))


def nvfp4_get_device_status(stream=None):
    return lib().nvfp4_get_device_status(_s(stream))


def nvfp4_status_string(status):
    return lib().nvfp4_status_string(status).decode()


def nvfp4_debug_scale_recipe_check(counters, mismatch, stream=None):
    _ok("nvfp4_debug_scale_recipe_check",
        lib().nvfp4_debug_scale_recipe_check(_p(counters), _p(mismatch), _s(stream)))


def nvfp4_debug_cvt_probe(first, last, counters, stream=None):
    _ok("nvfp4_debug_cvt_probe", lib().nvfp4_debug_cvt_probe(_p(first), _p(last), _p(counters),
                                                            _s(stream)))


def nvfp4_debug_wait_timeout(timeout_ns, stream=None):
    _ok("nvfp4_debug_wait_timeout", lib().nvfp4_debug_wait_timeout(timeout_ns, _s(stream)))


def nvfp4_debug_set_gemm_wait_limit(limit_ns):
    _ok("nvfp4_debug_set_gemm_wait_limit", lib().nvfp4_debug_set_gemm_wait_limit(limit_ns))


# ---------------------------------------------------------------------------
# Helpers that allocate outputs with torch and call the entry points above
# ---------------------------------------------------------------------------

def _u8(n, dev):
    return torch.empty(n, dtype=torch.uint8, device=dev)


class Workspace:
    """Caller-owned scratch buffer reused across calls on one stream."""

    def __init__(self, device, nbytes=0):
        self.device = device
        self.buf = _u8(max(int(nbytes), 256), device)

    def get(self, nbytes):
        if self.buf.numel() < nbytes:
            self.buf = _u8(int(nbytes), self.device)
        return self.buf


def quantize(x, gather=None, rows_out=None, mode="per_token", column_copy=False, workspace=None,
             stream=None):
    """Quantize the rows of a bf16 [rows, K] CUDA tensor; returns a dict of
    device tensors q [rows_out, K/2] uint8, sf (swizzled bytes), s [rows_out]
    float32, and with column_copy q_col / sf_col / s_col."""
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 2
    rows_in, K = x.shape
    ld = x.stride(0)
    assert x.stride(1) == 1
    if gather is not None:
        rows_out = gather.numel() if rows_out is None else rows_out
    elif rows_out is None:
        rows_out = rows_in
    dev = x.device
    out = dict(rows=rows_out, cols=K,
               q=_u8((rows_out, K // 2), dev), sf=_u8(nvfp4_sf_bytes(rows_out, K), dev),
               s=torch.empty(rows_out, dtype=torch.float32, device=dev))
    qc = sfc = sc = None
    if column_copy:
        qc = _u8((K, rows_out // 2), dev)
        sfc = _u8(nvfp4_sf_bytes(K, rows_out), dev)
        sc = torch.empty(1, dtype=torch.float32, device=dev)
        out.update(q_col=qc, sf_col=sfc, s_col=sc)
    m = PER_TENSOR if mode == "per_tensor" else PER_TOKEN
    ws = None
    wsb = 0
    if column_copy or m == PER_TENSOR:
        wsb = nvfp4_quantize_workspace_bytes()
        ws = (workspace or Workspace(dev)).get(wsb)
    nvfp4_quantize_per_token(x, rows_in, K, ld, gather, rows_out, m, out["q"], out["sf"], out["s"],
                             qc, sfc, sc, ws, wsb, stream)
    return out


def gemm(a, b, out=None, stream=None):
    """Y = a @ b^T (bf16) from two quantize() results (a: [M, K], b: [N, K])."""
    M, K = a["rows"], a["cols"]
    N = b["rows"]
    assert b["cols"] == K
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=a["q"].device)
    nvfp4_gemm(a["q"], a["sf"], a["s"], M, b["q"], b["sf"], b["s"], N, K, y, y.stride(0), stream)
    return y


def quantize_pair(x, w, column_copy=False, workspace=None, stream=None):
    """Per-token quantization of an activation x [rows_x, K] (optionally with its
    column-wise copy) and a weight w [rows_w, K] in one launch; returns two
    dicts shaped like quantize()'s."""
    assert x.dtype == torch.bfloat16 and w.dtype == torch.bfloat16 and x.shape[1] == w.shape[1]
    assert (x.shape[0] == 0 or x.stride(1) == 1) and (w.shape[0] == 0 or w.stride(1) == 1)
    K = x.shape[1]
    ld_x = x.stride(0) if x.shape[0] > 0 else K
    ld_w = w.stride(0) if w.shape[0] > 0 else K
    dev = x.device

    def outs(rows):
        return dict(rows=rows, cols=K, q=_u8((rows, K // 2), dev), sf=_u8(nvfp4_sf_bytes(rows, K), dev),
                    s=torch.empty(rows, dtype=torch.float32, device=dev))
    ox, ow = outs(x.shape[0]), outs(w.shape[0])
    qc = sfc = sc = ws = None
    wsb = 0
    if column_copy:
        qc = _u8((K, x.shape[0] // 2), dev)
        sfc = _u8(nvfp4_sf_bytes(K, x.shape[0]), dev)
        sc = torch.empty(1, dtype=torch.float32, device=dev)
        ox.update(q_col=qc, sf_col=sfc, s_col=sc)
        wsb = nvfp4_quantize_workspace_bytes()
        ws = (workspace or Workspace(dev)).get(wsb)
    nvfp4_quantize_per_token_pair(x, x.shape[0], ld_x, ox["q"], ox["sf"], ox["s"], qc, sfc, sc,
                                  w, w.shape[0], ld_w, ow["q"], ow["sf"], ow["s"], K, ws, wsb, stream)
    return ox, ow


def _operand(qres, column):
    if column:
        return qres["q_col"], qres["sf_col"], qres["s_col"], 0, qres["cols"], qres["rows"]
    return qres["q"], qres["sf"], qres["s"], 1, qres["rows"], qres["cols"]


def gemm_ex(a, b, a_column=False, b_column=False, out=None, stream=None):
    """Y = A B^T where A / B is a quantize() result's row-wise copy, or with
    *_column=True its column-wise copy (transposed operand, one outer scale)."""
    aq, asf, as_, apr, M, K = _operand(a, a_column)
    bq, bsf, bs, bpr, N, Kb = _operand(b, b_column)
    assert K == Kb
    y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    nvfp4_gemm_ex(aq, asf, as_, apr, M, bq, bsf, bs, bpr, N, K, y, y.stride(0), stream)
    return y


def gemm_dgrad(dy, w, out=None, stream=None):
    """dX [M, K] = dY [M, N] W [N, K]: dY's rows x W's column-wise copy."""
    return gemm_ex(dy, w, b_column=True, out=out, stream=stream)


def gemm_wgrad(dy, x, out=None, stream=None):
    """dW [N, K] = dY^T X: dY's and X's column-wise copies."""
    return gemm_ex(dy, x, a_column=True, b_column=True, out=out, stream=stream)


def moe_permute(topk_ids, num_experts, row_align=128, workspace=None, stream=None):
    T, k = topk_ids.shape
    dev = topk_ids.device
    cap = nvfp4_moe_capacity(T, k, num_experts, row_align)
    off = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    gather = torch.empty(cap, dtype=torch.int32, device=dev)
    dst = torch.empty((T, k), dtype=torch.int32, device=dev)
    wsb = nvfp4_moe_permute_workspace_bytes(T, k, num_experts)
    ws = (workspace or Workspace(dev)).get(wsb)
    nvfp4_moe_permute(topk_ids, T, k, num_experts, row_align, off, gather, cap, dst, ws, wsb, stream)
    return dict(offsets=off, gather=gather, dst=dst, capacity=cap)


def quantize_experts(w, stream=None):
    """Quantize stacked expert weights w [E, N, K] (bf16) per output row into the
    grouped GEMM's weight format: q [E, N, K/2], sf (E blocks of
    nvfp4_sf_bytes(N, K) bytes), s [E, N]."""
    E, N, K = w.shape
    dev = w.device
    sfb = nvfp4_sf_bytes(N, K)
    q = _u8((E, N, K // 2), dev)
    sf = _u8(E * sfb, dev)
    s = torch.empty((E, N), dtype=torch.float32, device=dev)
    flat = w.reshape(E * N, K)
    if N % 128 == 0:
        # 128-row scale tiles never straddle experts: one call lays out every block
        nvfp4_quantize_per_token(flat, E * N, K, K, None, E * N, PER_TOKEN, q, sf, s, stream=stream)
    else:
        for e in range(E):
            nvfp4_quantize_per_token(flat[e * N:(e + 1) * N], N, K, K, None, N, PER_TOKEN, q[e],
                                     sf.data_ptr() + e * sfb, s[e], stream=stream)
    return dict(rows=N, cols=K, experts=E, q=q, sf=sf, s=s)


def grouped_gemm(a, expert_offsets, num_experts, b_q, b_sf, b_s, N, K, out=None, stream=None):
    rows = a["rows"]
    y = out if out is not None else torch.empty((rows, N), dtype=torch.bfloat16, device=a["q"].device)
    nvfp4_grouped_gemm(a["q"], a["sf"], a["s"], rows, expert_offsets, num_experts, b_q, b_sf, b_s,
                       N, K, y, stream)
    return y


def grouped_gemm_swiglu(a, expert_offsets, num_experts, b_q, b_sf, b_s, ffn, K, out=None, stream=None):
    """h [rows, ffn] bf16 = bf16(silu(g) u) of the grouped fc1 product whose
    first ffn columns are the gate g and the next ffn the up projection u."""
    rows = a["rows"]
    h = out if out is not None else torch.empty((rows, ffn), dtype=torch.bfloat16, device=a["q"].device)
    nvfp4_grouped_gemm_swiglu(a["q"], a["sf"], a["s"], rows, expert_offsets, num_experts, b_q, b_sf, b_s, ffn, K,
                              h, stream)
    return h


def moe_combine(y2, dst_rows, weights, out=None, stream=None):
    """bf16 [tokens, hidden]: sum_j weights[t, j] * y2[dst_rows[t, j]] (binary32, slot order)."""
    tokens, topk = weights.shape
    hidden = y2.shape[1]
    o = out if out is not None else torch.empty((tokens, hidden), dtype=torch.bfloat16, device=y2.device)
    nvfp4_moe_combine(y2, y2.shape[0], y2.stride(0), dst_rows, weights, tokens, topk, hidden, o, o.stride(0),
                      stream)
    return o


def dequantize(qres, column=False, out=None, stream=None):
    """bf16 values of a quantize() result: the row-wise copy [rows, cols], or
    with column=True the column-wise copy [cols, rows] (one per-tensor scale)."""
    if column:
        q, sf, s = qres["q_col"], qres["sf_col"], qres["s_col"]
        rows, cols, per_row = qres["cols"], qres["rows"], 0
    else:
        q, sf, s = qres["q"], qres["sf"], qres["s"]
        rows, cols, per_row = qres["rows"], qres["cols"], 1
    y = out if out is not None else torch.empty((rows, cols), dtype=torch.bfloat16, device=q.device)
    nvfp4_dequantize(q, sf, s, per_row, rows, cols, y, y.stride(0), stream)
    return y


def moe_gather_quantized(qres, gather, offsets=None, stream=None):
    """Rows of a per-token quantize() result scattered to the routed layout
    (row r = source row gather[r], zero row where gather[r] < 0).  offsets, the
    permute's expert offsets, only order the work (token-window order)."""
    rows_out = gather.shape[0]
    cols = qres["cols"]
    dev = qres["q"].device
    out = dict(rows=rows_out, cols=cols, q=_u8((rows_out, cols // 2), dev),
               sf=_u8(nvfp4_sf_bytes(rows_out, cols), dev),
               s=torch.empty(rows_out, dtype=torch.float32, device=dev))
    num_experts = 0 if offsets is None else offsets.numel() - 1
    nvfp4_moe_gather_quantized(qres["q"], qres["sf"], qres["s"], qres["rows"], cols, gather, rows_out, offsets,
                               num_experts, out["q"], out["sf"], out["s"], stream)
    return out


def mxfp8_quantize(x, column_copy=False, stream=None):
    """MXFP8 of bf16 x [rows, cols]: q [rows, cols] E4M3 codes (uint8) and the
    swizzled E8M0 scales sf; with column_copy also q_col [cols, rows] and
    sf_col, the 32x1-block copy of X^T."""
    rows, cols = x.shape
    dev = x.device
    out = dict(rows=rows, cols=cols, q=_u8((rows, cols), dev), sf=_u8(nvfp4_mxfp8_sf_bytes(rows, cols), dev))
    if column_copy:
        out.update(q_col=_u8((cols, rows), dev), sf_col=_u8(nvfp4_mxfp8_sf_bytes(cols, rows), dev))
    nvfp4_mxfp8_quantize(x, rows, cols, x.stride(0), out["q"], out["sf"], out.get("q_col"), out.get("sf_col"),
                         stream)
    return out


def mxfp8_dequantize(qres, column=False, out=None, stream=None):
    """bf16 values of an mxfp8_quantize() result (column=True: the X^T copy)."""
    if column:
        q, sf, rows, cols = qres["q_col"], qres["sf_col"], qres["cols"], qres["rows"]
    else:
        q, sf, rows, cols = qres["q"], qres["sf"], qres["rows"], qres["cols"]
    y = out if out is not None else torch.empty((rows, cols), dtype=torch.bfloat16, device=q.device)
    nvfp4_mxfp8_dequantize(q, sf, rows, cols, y, y.stride(0), stream)
    return y


def swiglu_quantize(y1, ffn, row_count=None, want_h=False, stream=None):
    rows = y1.shape[0]
    dev = y1.device
    out = dict(rows=rows, cols=ffn, q=_u8((rows, ffn // 2), dev),
               sf=_u8(nvfp4_sf_bytes(rows, ffn), dev),
               s=torch.empty(rows, dtype=torch.float32, device=dev))
    h = torch.empty((rows, ffn), dtype=torch.bfloat16, device=dev) if want_h else None
    nvfp4_swiglu_quantize(y1, rows, ffn, y1.stride(0), row_count, out["q"], out["sf"], out["s"], h,
                          stream)
    if want_h:
        out["h"] = h
    return out


def get_device_status(stream=None):
    return nvfp4_get_device_status(stream)
