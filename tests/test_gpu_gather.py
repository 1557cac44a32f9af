"""The permutation fused into GEMM1 (the next item of the hot-path table:
gather the token rows in the GEMM's operand load instead of writing and
re-reading x_perm).  The fused path computes exactly what the unfused one
does -- same rows, same tiles, same arithmetic -- so every output is compared
bit for bit with moe_permute + moe_grouped_ffn (whose parity with the oracle
the kernel tests establish), in every GEMM execution mode, bf16 and e4m3; the
layer with MOE_GATHER=1 against the layer with the row copy."""
import numpy as np
import pytest
import torch

from helpers import assert_close, bits, f64, random_ids
from oracle import oracle as O
from test_gpu_kernels import FFN_MODES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _inputs(N, D, E, K, Dff, act, seed, skew=None):
    gen = torch.Generator().manual_seed(seed)
    ids = random_ids(N, E, K, gen, skew).cuda()
    x = torch.randn((N, D), generator=gen).to(torch.bfloat16).cuda()
    w1 = (torch.randn((E, Dff, D), generator=gen) * D ** -0.5).to(torch.bfloat16).cuda()
    w3 = (torch.randn((E, Dff, D), generator=gen) * D ** -0.5).to(torch.bfloat16).cuda() if act == 1 else None
    w2 = (torch.randn((E, D, Dff), generator=gen) * Dff ** -0.5).to(torch.bfloat16).cuda()
    return ids, x, w1, w3, w2


GATHER_CASES = [
    (300, 128, 8, 2, 256, 1, None),
    (300, 128, 8, 2, 256, 0, None),
    (777, 256, 16, 4, 128, 1, 1.5),       # skewed: long and empty segments
    (5, 512, 64, 8, 768, 1, None),        # decode-sized: swapped operands, split-K
    (2000, 256, 4, 2, 256, 1, None),      # CTA pairs in auto mode
    (64, 1024, 2, 1, 512, 0, None),       # few tiles: split-K of the SiLU GEMM1
]


@pytest.mark.parametrize("N,D,E,K,Dff,act,skew", GATHER_CASES)
@pytest.mark.parametrize("mode", list(FFN_MODES) + ["pair"])
def test_gathered_ffn_equals_unfused_bitwise(moe, N, D, E, K, Dff, act, skew, mode, monkeypatch):
    for k, v in FFN_MODES.get(mode, {"MOE_PAIR_GEMM": "1"}).items():
        monkeypatch.setenv(k, v)
    ids, x, w1, w3, w2 = _inputs(N, D, E, K, Dff, act, seed=N + D + E + act)
    off, ps, ip, xp = moe.moe_permute(x, ids, E)
    off2, ps2, ip2 = moe.moe_permute_indices(ids, E)
    assert torch.equal(off, off2) and torch.equal(ps, ps2) and torch.equal(ip, ip2)
    h0, y0 = moe.moe_grouped_ffn(xp, off, w1, w3, w2, act)
    ws = moe.workspace("ffn", N * K, D, E, 1, Dff)
    h1, y1 = moe.moe_grouped_ffn_gathered(x, ps2, off2, w1, w3, w2, act, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(h0, h1) and torch.equal(y0, y1)


@pytest.mark.parametrize("N,D,E,K,Dff,act,skew", [c for c in GATHER_CASES if c[1] % 128 == 0 and c[4] % 128 == 0])
@pytest.mark.parametrize("mode", ["auto", "one_n64", "swap", "pair"])
def test_gathered_e4m3_ffn_equals_unfused_bitwise(moe, N, D, E, K, Dff, act, skew, mode, monkeypatch):
    for k, v in FFN_MODES.get(mode, {"MOE_PAIR_GEMM": "1"}).items():
        monkeypatch.setenv(k, v)
    ids, x, w1, w3, w2 = _inputs(N, D, E, K, Dff, act, seed=N + D + E + act + 1)
    qw = moe.quantize_experts_e4m3(w1, w3, w2)
    xq, sx = moe.moe_quantize_e4m3(x)
    off, ps, ip, xqp = moe.moe_permute_e4m3(xq, ids, E)
    r0 = moe.moe_grouped_ffn_e4m3(xqp, sx, ps, off, qw["w1q"], qw["s1"], qw["w3q"], qw["s3"], qw["w2q"], qw["s2"],
                                  act)
    ws = moe.workspace("ffn", N * K, D, E, 1, Dff)
    r1 = moe.moe_grouped_ffn_e4m3_gathered(xq, sx, ps, off, qw["w1q"], qw["s1"], qw["w3q"], qw["s3"], qw["w2q"],
                                           qw["s2"], act, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    for a, b in zip(r0, r1):
        assert torch.equal(a, b)


def test_gathered_ffn_flags_bad_source_rows(moe):
    N, D, E, K, Dff = 40, 128, 4, 2, 128
    ids, x, w1, w3, w2 = _inputs(N, D, E, K, Dff, 1, seed=9)
    off, ps, _ = moe.moe_permute_indices(ids, E)
    ps = ps.clone()
    ps[7] = N + 3            # a source row outside x: skipped and flagged
    ws = moe.workspace("ffn", N * K, D, E, 1, Dff)
    moe.moe_grouped_ffn_gathered(x, ps, off, w1, w3, w2, 1, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_BOUNDS


@pytest.mark.parametrize("precision", ["bf16", "e4m3"])
@pytest.mark.parametrize("N,D,E,K,Dff", [(300, 128, 32, 8, 128), (2048, 256, 4, 2, 256), (3, 256, 16, 4, 256)])
def test_layer_fused_equals_unfused_bitwise(moe, N, D, E, K, Dff, precision, monkeypatch):
    from mixture_experts_layer_02_gb300 import synth
    monkeypatch.setenv("MOE_LAYER_DECODE", "0")   # small N: compare the chain of launches, gathered or not
    wl = synth.Workload("g", N, D, E, K, Dff, 1, 1, 0.0)
    inp = {k: (None if v is None else v.cuda()) for k, v in synth.make_inputs(wl, seed=5).items()}
    outs = []
    for flag in ("1", "0"):
        monkeypatch.setenv("MOE_GATHER", flag)
        if precision == "bf16":
            outs.append(moe.moe_layer_forward(inp["x"], inp["w_gate"], None, inp["w1"], inp["w3"], inp["w2"],
                                              K, 1, 1))
        else:
            qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
            outs.append(moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], None, qw, K, 1, 1))
    assert torch.equal(outs[0], outs[1])
