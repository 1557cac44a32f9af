"""The allocation-free permutation entry point, checked against moe_permute.

moe_permute_static_scratch serves callers that cannot allocate device memory
while the layer runs (engines that plan every buffer up front and forbid
allocation during execution).  It must produce exactly what the workspace
version produces.  Two calls in a row with different sizes check that the
library-owned scratch left behind by one call does not leak into the next.
This file is collected last so that a failure here never hides the others.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _inputs(N, E, K, D, seed):
    g = torch.Generator().manual_seed(seed)
    ids = torch.topk(torch.rand((N, E), generator=g), K, dim=1).indices.to(torch.int32)
    x = torch.randn((N, D), generator=g).to(torch.bfloat16)
    return x.cuda(), ids.cuda()


def test_static_scratch_permute_matches_workspace_permute(moe):
    # larger call first, then a smaller one over the same shared scratch
    for N, E, K, D, seed in [(4096, 256, 8, 256, 1), (333, 60, 6, 128, 2)]:
        x, ids = _inputs(N, E, K, D, seed)
        ref = moe.moe_permute(x, ids, E)
        got = moe.moe_permute_static_scratch(x, ids, E)
        torch.cuda.synchronize()
        for name, a, b in zip(("expert_offsets", "perm_src", "inv_perm", "x_perm"), got, ref):
            assert torch.equal(a, b), name


def test_static_scratch_rejects_sizes_beyond_its_maximum(moe):
    lib = moe.load()
    p = ctypes.c_void_p
    # E * ceil(N/16) + E > 2^20: refused on the host, nothing is launched
    st = lib.moe_permute_static_scratch(p(4096), p(8192), 1 << 16, 64, 1024, 8, p(256), p(512), p(768),
                                        p(1024), None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert b"static maximum" in lib.moe_last_error_detail()
