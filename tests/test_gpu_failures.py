"""Failure detection without a GPU fault: a bounded pipeline wait that runs
out reports MOE_ERR_DEVICE_TIMEOUT through the workspace error word, the CTA
returns (no trap, no hang), and the CUDA context stays usable."""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _case():
    g = torch.Generator().manual_seed(77)
    counts = [130, 5, 0, 64]
    E, D, Dff = len(counts), 128, 128
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32).cuda()
    xp = torch.randn((sum(counts), D), generator=g).to(torch.bfloat16).cuda()
    w1 = (torch.randn((E, Dff, D), generator=g) * D ** -0.5).to(torch.bfloat16).cuda()
    w3 = (torch.randn((E, Dff, D), generator=g) * D ** -0.5).to(torch.bfloat16).cuda()
    w2 = (torch.randn((E, D, Dff), generator=g) * Dff ** -0.5).to(torch.bfloat16).cuda()
    return xp, off, w1, w3, w2


def test_withheld_load_times_out_and_context_survives(moe):
    xp, off, w1, w3, w2 = _case()
    ref_h, ref_y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU)
    torch.cuda.synchronize()
    ws = moe.workspace("ffn", xp.shape[0], xp.shape[1], w1.shape[0], 1, w1.shape[1])
    moe.set_debug_flags(ws, 1)   # the first operand load of CTA 0 is never issued
    t0 = time.time()
    moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    status = moe.read_device_error(ws)
    elapsed = time.time() - t0
    assert status == moe.MOE_ERR_DEVICE_TIMEOUT
    assert elapsed < 30.0
    # the context is intact: clear the header and compute again
    moe.clear_device_error(ws)
    h, y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(h, ref_h) and torch.equal(y, ref_y)


def test_withheld_load_in_the_mixed_pair_kernel(moe, monkeypatch):
    """The same on the mixed CTA-pair kernel (hot pair tiles and cold
    weight-streaming tiles in one launch): the stalled pair gives up, the
    peer CTA's exchange waits give up too, and the context stays usable."""
    monkeypatch.setenv("MOE_PAIR_GEMM", "1")
    monkeypatch.setenv("MOE_SWAP_GEMM", "0")
    monkeypatch.setenv("MOE_PAIR_COLD_ROWS", "64")
    g = torch.Generator().manual_seed(78)
    counts = [300, 5, 0, 64, 1, 40, 513, 2, 90, 7, 0, 33, 12, 260, 3, 9]
    E, D, Dff = len(counts), 256, 256
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32).cuda()
    xp = torch.randn((sum(counts), D), generator=g).to(torch.bfloat16).cuda()
    w1 = (torch.randn((E, Dff, D), generator=g) * D ** -0.5).to(torch.bfloat16).cuda()
    w3 = (torch.randn((E, Dff, D), generator=g) * D ** -0.5).to(torch.bfloat16).cuda()
    w2 = (torch.randn((E, D, Dff), generator=g) * Dff ** -0.5).to(torch.bfloat16).cuda()
    ref_h, ref_y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU)
    torch.cuda.synchronize()
    ws = moe.workspace("ffn", xp.shape[0], D, E, 1, Dff)
    moe.set_debug_flags(ws, 1)
    t0 = time.time()
    moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    status = moe.read_device_error(ws)
    assert status == moe.MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30.0
    moe.clear_device_error(ws)
    h, y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(h, ref_h) and torch.equal(y, ref_y)
