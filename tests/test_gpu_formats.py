"""The device's E2M1 / E4M3 conversions against the oracle's encoders, over all
2^31 non-negative float32 patterns (and, by the symmetry counter, the negative
half for E2M1), plus the library's bounded-wait failure path.

Both encoders are non-decreasing step functions of the bit pattern of a
non-negative float (the GPU's monotonicity is counted by the probe, the
oracle's follows from nearest-value search), so equal codes at every step edge
the GPU reports, and one pattern either side of it, mean equal codes for every
input.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _codes_at(orc, patterns, which):
    x = np.array(patterns, np.uint32).view(np.float32)
    return orc.e2m1_encode(x) if which == "e2m1" else orc.e4m3_encode(x)


def test_exhaustive_cvt_matches_oracle(nv, orc):
    first = torch.empty(144, dtype=torch.int32, device="cuda")
    last = torch.empty(144, dtype=torch.int32, device="cuda")
    cnt = torch.empty(4, dtype=torch.int32, device="cuda")
    nv.nvfp4_debug_cvt_probe(first, last, cnt)
    torch.cuda.synchronize()
    first = first.cpu().numpy().view(np.uint32)
    last = last.cpu().numpy().view(np.uint32)
    cnt = cnt.cpu().numpy().view(np.uint32)
    assert cnt.tolist() == [0, 0, 0, 0], cnt      # monotone, sign-symmetric, no NaN codes
    for which, base, ncodes in (("e2m1", 0, 8), ("e4m3", 16, 127)):
        present = [c for c in range(ncodes) if first[base + c] != 0xFFFFFFFF]
        assert present == list(range(ncodes)), (which, present)
        assert first[base] == 0 and last[base + ncodes - 1] == 0x7F800000
        for c in range(ncodes):
            f, l = int(first[base + c]), int(last[base + c])
            assert f <= l
            assert list(_codes_at(orc, [f, l], which)) == [c, c], (which, c, hex(f), hex(l))
            if c > 0:
                assert int(last[base + c - 1]) + 1 == f
                assert _codes_at(orc, [f - 1], which)[0] == c - 1
            if c + 1 < ncodes:
                assert _codes_at(orc, [l + 1], which)[0] == c + 1
    # E4M3 NaN code never produced
    assert first[16 + 127] == 0xFFFFFFFF


def test_bounded_wait_times_out_and_context_survives(nv):
    assert nv.nvfp4_get_device_status() == 0
    nv.nvfp4_debug_wait_timeout(50_000_000)        # 50 ms, nothing ever arrives
    assert nv.nvfp4_get_device_status() == 6      # NVFP4_ERR_TIMEOUT
    assert nv.nvfp4_get_device_status() == 0      # cleared
    x = torch.randn(64, 256, device="cuda").to(torch.bfloat16)
    out = nv.quantize(x)
    torch.cuda.synchronize()
    assert out["s"].abs().sum().item() > 0
