"""The non-allocating routing permute (nvfp4_moe_permute_noalloc), for callers
that cannot call cudaMalloc where they route tokens (device memory owned by
another allocator, allocation-free decode loops).  It must produce exactly what the
allocating nvfp4_moe_permute produces, on consecutive calls that reuse the
library's fixed scratch array, and refuse sizes past that array.  This file is
collected last so a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

from nvfp4_precision_rl_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _outputs(nv, tokens, topk, experts):
    cap = nv.nvfp4_moe_capacity(tokens, topk, experts, 128)
    return (torch.empty(experts + 1, dtype=torch.int32, device="cuda"),
            torch.empty(cap, dtype=torch.int32, device="cuda"),
            torch.empty((tokens, topk), dtype=torch.int32, device="cuda"), cap)


@pytest.mark.parametrize("T,E,k", [(4096, 128, 8), (37, 8, 2), (65536, 128, 8)])
def test_noalloc_permute_matches_allocating_permute(nv, T, E, k):
    ids = torch.from_numpy(W.route_topk(np.random.default_rng(T + k), T, E, k)).cuda()
    ref = nv.moe_permute(ids, E)
    torch.cuda.synchronize()
    for _ in range(2):   # two calls in a row share the scratch array
        off, gather, dst, cap = _outputs(nv, T, k, E)
        nv.nvfp4_moe_permute_noalloc(ids, T, k, E, 128, off, gather, cap, dst)
        torch.cuda.synchronize()
        assert nv.nvfp4_get_device_status() == 0
        assert torch.equal(off, ref["offsets"])
        assert torch.equal(gather, ref["gather"])
        assert torch.equal(dst, ref["dst"])


def test_noalloc_permute_rejects_sizes_past_its_scratch(nv):
    T, k, E = 300_000, 8, 128          # 2.4 M routed pairs: histograms exceed 1 MiB
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    off, gather, dst, cap = _outputs(nv, T, k, E)
    with pytest.raises(nv.NVFP4Error) as err:
        nv.nvfp4_moe_permute_noalloc(ids, T, k, E, 128, off, gather, cap, dst)
    assert err.value.status == 8        # NVFP4_ERR_WORKSPACE
