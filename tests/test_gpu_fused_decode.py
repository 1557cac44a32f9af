"""The decode-sized SwiGLU FFN in one persistent launch (GEMM1 + SwiGLU and
GEMM2, split partials summed by the last split of each tile, GEMM2 items of
an expert waiting until its h is written).  It sums the same fp32 partials in
the same order as the separate launches, so h and y must equal the unfused
swapped-operand path (MOE_FUSED_DECODE=0) bit for bit; the kernel tests'
"swap" mode and the full-size decode workloads check it against the oracle."""
import time

import numpy as np
import pytest
import torch

from helpers import assert_close, bits, random_ids
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _case(moe, N, D, E, K, Dff, seed):
    gen = torch.Generator().manual_seed(seed)
    ids = random_ids(N, E, K, gen).cuda()
    x = torch.randn((N, D), generator=gen).to(torch.bfloat16).cuda()
    w1 = (torch.randn((E, Dff, D), generator=gen) * D ** -0.5).to(torch.bfloat16).cuda()
    w3 = (torch.randn((E, Dff, D), generator=gen) * D ** -0.5).to(torch.bfloat16).cuda()
    w2 = (torch.randn((E, D, Dff), generator=gen) * Dff ** -0.5).to(torch.bfloat16).cuda()
    off, ps, ip, xp = moe.moe_permute(x, ids, E)
    return x, off, xp, w1, w3, w2


DECODE_CASES = [
    (1, 2048, 128, 8, 768),      # one token: 8 experts, split GEMM1 and GEMM2
    (8, 2048, 128, 8, 768),
    (32, 2048, 128, 8, 768),
    (256, 2048, 128, 8, 768),    # every expert, 16 rows each
    (3, 256, 16, 4, 256),
    (40, 512, 4, 2, 1024),       # few experts with 20 rows: 32-token tiles
]


@pytest.mark.parametrize("N,D,E,K,Dff", DECODE_CASES)
def test_fused_decode_equals_separate_launches(moe, N, D, E, K, Dff, monkeypatch):
    x, off, xp, w1, w3, w2 = _case(moe, N, D, E, K, Dff, seed=N + E)
    ws = moe.workspace("ffn", N * K, D, E, 1, Dff)
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")   # at every size, also below the default threshold
    h1, y1 = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    monkeypatch.setenv("MOE_FUSED_DECODE", "0")
    h0, y0 = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(h0, h1) and torch.equal(y0, y1)


@pytest.mark.parametrize("N,D,E,K,Dff", DECODE_CASES[:2] + DECODE_CASES[4:])
def test_fused_decode_matches_oracle(moe, N, D, E, K, Dff, monkeypatch):
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")
    x, off, xp, w1, w3, w2 = _case(moe, N, D, E, K, Dff, seed=3 * N + E)
    h, y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU)
    offn = off.cpu().numpy()
    hg = bits(h)
    h_ref = np.zeros((N * K, Dff))
    y_ref = np.zeros((N * K, D))
    for e in range(E):
        a, b = int(offn[e]), int(offn[e + 1])
        if a < b:
            h_ref[a:b] = O.expert_up(bits(xp[a:b]), bits(w1[e]), bits(w3[e]), O.ACT_SWIGLU)
            y_ref[a:b] = O.expert_down(hg[a:b], bits(w2[e]))
    assert_close(O.bf16_to_f64(hg), h_ref, "h")
    assert_close(O.bf16_to_f64(bits(y)), y_ref, "y_perm")


def test_fused_decode_is_deterministic(moe):
    x, off, xp, w1, w3, w2 = _case(moe, 32, 2048, 128, 8, 768, seed=11)
    a = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU)
    b = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fused_decode_withheld_load_times_out_and_context_survives(moe, monkeypatch):
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")
    x, off, xp, w1, w3, w2 = _case(moe, 8, 2048, 128, 8, 768, seed=5)
    ref_h, ref_y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU)
    torch.cuda.synchronize()
    ws = moe.workspace("ffn", xp.shape[0], xp.shape[1], w1.shape[0], 1, w1.shape[1])
    moe.set_debug_flags(ws, 1)   # the first operand load of CTA 0 is never issued
    t0 = time.time()
    moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    status = moe.read_device_error(ws)
    assert status == moe.MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30.0
    moe.clear_device_error(ws)
    h, y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(h, ref_h) and torch.equal(y, ref_y)
