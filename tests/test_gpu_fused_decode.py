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
    (1, 2048, 128, 8, 768),      # one token: 8 experts
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


# k-splits pinned (MOE_FFN_SPLITS=s1,s2): fp32 partials of every split, the
# last split of each tile summing them in split order, in both paths
SPLIT_CASES = [((1, 2048, 128, 8, 768), "3,2"), ((1, 2048, 128, 8, 768), "4,4"), ((8, 2048, 128, 8, 768), "2,3")]


@pytest.mark.parametrize("case,splits", SPLIT_CASES)
def test_fused_decode_split_equals_separate_launches(moe, case, splits, monkeypatch):
    N, D, E, K, Dff = case
    x, off, xp, w1, w3, w2 = _case(moe, N, D, E, K, Dff, seed=N + E + 1)
    ws = moe.workspace("ffn", N * K, D, E, 1, Dff)
    monkeypatch.setenv("MOE_FFN_SPLITS", splits)
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")
    h1, y1 = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    monkeypatch.setenv("MOE_FUSED_DECODE", "0")
    h0, y0 = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(h0, h1) and torch.equal(y0, y1)
    # and the split sums agree with the unsplit path within rounding
    monkeypatch.setenv("MOE_FFN_SPLITS", "1,1")
    h2, y2 = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=ws)
    assert_close(O.bf16_to_f64(bits(y1)), O.bf16_to_f64(bits(y2)), "split vs unsplit y")


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


# ---- e4m3 operands: GEMM1 + SwiGLU, the h quantisation and GEMM2 in the same launch


def _case_e4m3(moe, N, D, E, K, Dff, seed, per_token):
    x, off, xp, w1, w3, w2 = _case(moe, N, D, E, K, Dff, seed)
    qw = moe.quantize_experts_e4m3(w1, w3, w2)
    xq, sx = moe.moe_quantize_e4m3(x)
    gen = torch.Generator().manual_seed(seed)
    ids = random_ids(N, E, K, gen).cuda()
    off, ps, ip, xqp = moe.moe_permute_e4m3(xq, ids, E)
    # token scales per token (through perm_src) or per permuted row
    scale, idx = (sx, ps) if per_token else (sx[ps.long()].contiguous(), None)
    return off, ps, xqp, scale, idx, qw


E4M3_CASES = DECODE_CASES + [(2, 2048, 128, 8, 768)]


@pytest.mark.parametrize("per_token", [True, False])
@pytest.mark.parametrize("N,D,E,K,Dff", E4M3_CASES)
def test_fused_decode_e4m3_equals_separate_launches(moe, N, D, E, K, Dff, per_token, monkeypatch):
    off, ps, xqp, scale, idx, qw = _case_e4m3(moe, N, D, E, K, Dff, N + 7 * E, per_token)
    ws = moe.workspace("ffn", N * K, D, E, 1, Dff)
    run = lambda: moe.moe_grouped_ffn_e4m3(xqp, scale, idx, off, qw["w1q"], qw["s1"], qw["w3q"], qw["s3"],
                                           qw["w2q"], qw["s2"], moe.ACT_SWIGLU, ws=ws)
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")
    fused = run()
    assert moe.read_device_error(ws) == moe.MOE_OK
    monkeypatch.setenv("MOE_FUSED_DECODE", "0")
    sep = run()
    assert moe.read_device_error(ws) == moe.MOE_OK
    for a, b, name in zip(fused, sep, ("h", "hq", "h_scale", "y_perm")):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("case,splits", SPLIT_CASES)
def test_fused_decode_e4m3_split_equals_separate_launches(moe, case, splits, monkeypatch):
    N, D, E, K, Dff = case
    off, ps, xqp, scale, idx, qw = _case_e4m3(moe, N, D, E, K, Dff, N + 3 * E, True)
    ws = moe.workspace("ffn", N * K, D, E, 1, Dff)
    run = lambda: moe.moe_grouped_ffn_e4m3(xqp, scale, idx, off, qw["w1q"], qw["s1"], qw["w3q"], qw["s3"],
                                           qw["w2q"], qw["s2"], moe.ACT_SWIGLU, ws=ws)
    monkeypatch.setenv("MOE_FFN_SPLITS", splits)
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")
    fused = [t.clone() for t in run()]
    assert moe.read_device_error(ws) == moe.MOE_OK
    monkeypatch.setenv("MOE_FUSED_DECODE", "0")
    sep = run()
    assert moe.read_device_error(ws) == moe.MOE_OK
    for a, b, name in zip(fused, sep, ("h", "hq", "h_scale", "y_perm")):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("N,D,E,K,Dff", [(8, 2048, 128, 8, 768), (3, 256, 16, 4, 256), (40, 512, 4, 2, 1024)])
def test_fused_decode_e4m3_matches_oracle(moe, N, D, E, K, Dff, monkeypatch):
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")
    off, ps, xqp, scale, idx, qw = _case_e4m3(moe, N, D, E, K, Dff, 5 * N + E, True)
    h, hq, hs, y = moe.moe_grouped_ffn_e4m3(xqp, scale, idx, off, qw["w1q"], qw["s1"], qw["w3q"], qw["s3"],
                                            qw["w2q"], qw["s2"], moe.ACT_SWIGLU)
    u8 = lambda t: t.detach().contiguous().cpu().numpy()
    sx_rows = u8(scale)[u8(ps)]
    g = O.grouped_ffn_e4m3(u8(xqp), sx_rows, u8(off), u8(qw["w1q"]), u8(qw["s1"]), u8(qw["w3q"]), u8(qw["s3"]),
                           u8(qw["w2q"]), u8(qw["s2"]), O.ACT_SWIGLU)
    assert_close(O.bf16_to_f64(bits(h)), g["h"], "h")
    # the codes of the GPU's own h are the oracle's quantisation of it, bit for bit
    r_hq, r_hs = O.quant_rows_e4m3(bits(h))
    assert np.array_equal(u8(hq), r_hq) and np.array_equal(u8(hs), r_hs)
    offn = u8(off)
    y_ref = np.zeros((N * K, D))
    for e in range(E):
        a, b = int(offn[e]), int(offn[e + 1])
        if a < b:
            y_ref[a:b] = O.expert_down_e4m3(r_hq[a:b], r_hs[a:b], u8(qw["w2q"][e]), u8(qw["s2"][e]))
    assert_close(O.bf16_to_f64(bits(y)), y_ref, "y_perm")


def test_fused_decode_e4m3_withheld_load_times_out_and_context_survives(moe, monkeypatch):
    monkeypatch.setenv("MOE_FUSED_DECODE", "1")
    off, ps, xqp, scale, idx, qw = _case_e4m3(moe, 8, 2048, 128, 8, 768, 9, True)
    ws = moe.workspace("ffn", xqp.shape[0], xqp.shape[1], 128, 1, 768)
    run = lambda: moe.moe_grouped_ffn_e4m3(xqp, scale, idx, off, qw["w1q"], qw["s1"], qw["w3q"], qw["s3"],
                                           qw["w2q"], qw["s2"], moe.ACT_SWIGLU, ws=ws)
    ref = [t.clone() for t in run()]
    torch.cuda.synchronize()
    moe.set_debug_flags(ws, 1)   # the first operand load of CTA 0 is never issued
    t0 = time.time()
    run()
    assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30.0
    moe.set_debug_flags(ws, 0)
    moe.clear_device_error(ws)
    out = run()
    assert moe.read_device_error(ws) == moe.MOE_OK
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
