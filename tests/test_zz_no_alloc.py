"""The allocation-free permutation entry point, against the oracle and against
moe_permute.

moe_permute_static_scratch serves callers that cannot allocate device memory
while the layer runs (engines that plan every buffer up front and forbid
allocation during execution).  It must give exactly what the oracle's
placement gives ("MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切",
第二层 范式 A Step 1) and what the workspace version gives.  Calls in a row
with different sizes, largest first, check that the library-owned scratch
left behind by one call does not leak into the next; every size here takes
the multi-launch path that uses that scratch (more than 4096 assignments).
This file is collected last so that a failure here never hides the others.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import bits
from oracle import oracle as O

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


def test_static_scratch_permute_matches_oracle_and_workspace_permute(moe):
    # (N, E, K, D): the documented maximum's neighbourhood first (16384 tokens,
    # 256 experts: 262,400 of the 1,048,576 scratch ints), then smaller calls
    # over the same shared scratch
    for N, E, K, D, seed in [(16384, 256, 8, 64, 1), (4096, 256, 8, 256, 2), (1000, 60, 6, 128, 3)]:
        assert N * K > 4096                       # the path that uses the scratch
        x, ids = _inputs(N, E, K, D, seed)
        got = moe.moe_permute_static_scratch(x, ids, E)
        ref = moe.moe_permute(x, ids, E)
        torch.cuda.synchronize()
        for name, a, b in zip(("expert_offsets", "perm_src", "inv_perm", "x_perm"), got, ref):
            assert torch.equal(a, b), name
        ids_h = ids.cpu().numpy()
        off = O.offsets(ids_h, E)
        perm_src, inv_perm = O.place(ids_h, off, E)
        assert np.array_equal(got[0].cpu().numpy(), off)
        assert np.array_equal(got[1].cpu().numpy(), perm_src)
        assert np.array_equal(got[2].cpu().numpy(), inv_perm)
        assert np.array_equal(bits(got[3]), O.gather_rows(bits(x), perm_src))


@pytest.mark.parametrize("N", [300, 1200])          # one-launch path and the scratch path
def test_static_scratch_skips_ids_outside_the_expert_range(moe, N):
    # the documented behaviour for bad ids: skipped, inv_perm = -1, and the
    # valid assignments placed exactly as if the bad ones were absent
    E, K, D = 40, 4, 64
    x, ids = _inputs(N, E, K, D, 5)
    ids_h = ids.cpu().numpy()
    bad = [(0, 1), (7, 0), (N // 2, 3), (N - 1, 2)]
    for (t, k), v in zip(bad, (E, -1, 1000, E + 7)):
        ids_h[t, k] = v
    ids = torch.as_tensor(ids_h).cuda()
    ps = torch.full((N * K,), -7, dtype=torch.int32, device="cuda")
    got = moe.moe_permute_static_scratch(x, ids, E, perm_src=ps)
    torch.cuda.synchronize()
    off, perm_src, inv_perm = (t.cpu().numpy() for t in got[:3])
    valid = (ids_h >= 0) & (ids_h < E)
    nvalid = int(valid.sum())
    assert nvalid == N * K - len(bad)
    # expected: stable placement, in (t, k) order, of the valid assignments only
    counts = np.bincount(ids_h[valid], minlength=E)
    exp_off = np.concatenate([[0], np.cumsum(counts)])
    assert np.array_equal(off, exp_off) and off[E] == nvalid
    fill = exp_off[:-1].copy()
    exp_inv = np.full((N, K), -1, np.int64)
    exp_src = np.empty(nvalid, np.int64)
    for t in range(N):
        for k in range(K):
            if valid[t, k]:
                r = fill[ids_h[t, k]]
                fill[ids_h[t, k]] += 1
                exp_inv[t, k] = r
                exp_src[r] = t
    assert np.array_equal(inv_perm, exp_inv)
    for t, k in bad:
        assert inv_perm[t, k] == -1
    assert np.array_equal(perm_src[:nvalid], exp_src)
    assert np.all(perm_src[nvalid:] == -7)             # rows past the valid ones are not written
    assert np.array_equal(bits(got[3][:nvalid]), bits(x)[exp_src])


def test_static_scratch_rejects_sizes_beyond_its_maximum(moe):
    # E * ceil(N/16) + E = 1024 * 1024 + 1024 > 2^20: refused on the host, with
    # real device buffers of the right sizes, so that a broken size check
    # would show as a failed assertion and never as a fault
    N, E, K, D = 16384, 1024, 8, 64
    x = torch.zeros((N, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((N, K), dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -5, dtype=torch.int32, device="cuda")
    ps = torch.empty(N * K, dtype=torch.int32, device="cuda")
    inv = torch.empty((N, K), dtype=torch.int32, device="cuda")
    xp = torch.empty((N * K, D), dtype=torch.bfloat16, device="cuda")
    lib = moe.load()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.moe_permute_static_scratch(p(x), p(ids), N, D, E, K, p(off), p(ps), p(inv), p(xp), None)
    torch.cuda.synchronize()
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert b"static maximum" in lib.moe_last_error_detail()
    assert torch.all(off == -5)                        # nothing was enqueued
    # the same sizes that moe_permute rejects are rejected here too (D not a
    # multiple of 64; buffers sized for D = 96 all the same)
    N, E, K, D = 64, 8, 2, 96
    x = torch.zeros((N, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((N, K), dtype=torch.int32, device="cuda")
    xp = torch.empty((N * K, D), dtype=torch.bfloat16, device="cuda")
    for fn in (lambda: lib.moe_permute_static_scratch(p(x), p(ids), N, D, E, K, p(off), p(ps), p(inv), p(xp),
                                                      None),
               lambda: lib.moe_permute(p(x), p(ids), N, D, E, K, p(off), p(ps), p(inv), p(xp), p(ps),
                                       ps.numel() * 4, None)):
        assert fn() == moe.MOE_ERR_INVALID_ARG
        assert b"D=96" in lib.moe_last_error_detail()
    torch.cuda.synchronize()
    assert torch.all(off == -5)
