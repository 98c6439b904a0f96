"""Shared helpers of the GPU parity tests (host-side comparison only)."""
import numpy as np
import torch


def to_dev(bits):
    """uint16 bf16 bits (numpy) -> torch.bfloat16 CUDA tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def host(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(t):
    """bf16 CUDA tensor -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


def assert_quant_equal(gpu, ref, rows=None, what="", col=False):
    """Bit-exact comparison of a GPU quantize() result with the oracle's."""
    kq, ksf, ks = ("q_col", "sf_col", "s_col") if col else ("q", "sf", "s")
    refsf = "sf_col_swz" if col else "sf_swz"
    gq, gsf, gs = host(gpu[kq]), host(gpu[ksf]), host(gpu[ks])
    rq, rsf, rs = ref[kq], ref[refsf], ref[ks]
    if rows is not None:
        gq, gs = gq[rows], gs[rows]
        rq, rs = rq[rows], rs[rows]
    bad = np.argwhere(gq != rq)
    assert bad.size == 0, f"{what}: {len(bad)} packed bytes differ, first at {bad[:5].tolist()}"
    assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32)), f"{what}: outer scales differ"
    if rows is None:
        badsf = np.nonzero(gsf != rsf)[0]
        assert badsf.size == 0, f"{what}: {badsf.size} scale bytes differ, first at {badsf[:8]}"


def bf16_ulp(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return 2.0 ** np.maximum(e - 7, -133)


def bf16_floor(y_ref):
    """Normwise relative error of rounding the exact result itself to bf16."""
    yr = torch.from_numpy(np.asarray(y_ref, np.float64)).to(torch.bfloat16).double().numpy()
    den = np.linalg.norm(y_ref)
    return float(np.linalg.norm(yr - y_ref) / den) if den > 0 else 0.0


def check_gemm(y_gpu, y_ref, absy, K, what=""):
    """GEMM tolerance (reading of the pages' "max relative error 2e-3 after bf16
    rounding"): (i) normwise relative error <= 2e-3, or, for outputs so small
    that bf16 rounding of the exact result alone exceeds that (a handful of
    elements), <= 1.25 x that rounding floor; (ii) every element within one bf16
    ulp of the exact value plus a 4 * K * 2^-24 FP32-summation allowance."""
    y_gpu = np.asarray(y_gpu, np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = bf16_ulp(y_ref) + 4.0 * K * 2.0 ** -24 * absy
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} elements out of bound; first {bad[:5].tolist()} "
                           f"gpu={y_gpu[tuple(bad[0])]} ref={y_ref[tuple(bad[0])]}")
    den = np.linalg.norm(y_ref)
    if den > 0:
        rel = np.linalg.norm(y_gpu - y_ref) / den
        gate = max(2e-3, 1.25 * bf16_floor(y_ref))
        assert rel <= gate, f"{what}: normwise relative error {rel:.3e} > {gate:.3e}"
    return float(np.max(err / np.maximum(np.abs(y_ref), 1e-30))) if y_ref.size else 0.0
