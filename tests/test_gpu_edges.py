"""Edge cases of the whole path: zero tokens through every entry point, the
largest expert count and K the limits allow on both router paths, and a
degenerate routing in which a bias sends every token to one expert."""
import numpy as np
import pytest
import torch

from helpers import WEIGHT_ATOL, assert_close, bits, f64, logits_bound, near_tie_mask
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).to(torch.bfloat16)


def test_zero_tokens_are_no_ops(moe):
    # N = 0 is a valid call of every entry point: MOE_OK, no device error,
    # expert_offsets all zero where a permutation is asked for
    D, E, K, Dff = 256, 16, 4, 256
    gen = torch.Generator().manual_seed(1)
    x = torch.empty((0, D), dtype=torch.bfloat16, device="cuda")
    wg = _bf16((E, D), gen, D ** -0.5).cuda()
    w1 = _bf16((E, Dff, D), gen, D ** -0.5).cuda()
    w3 = _bf16((E, Dff, D), gen, D ** -0.5).cuda()
    w2 = _bf16((E, D, Dff), gen, Dff ** -0.5).cuda()

    ids, w = moe.moe_route(x, wg, None, K, 0)
    assert ids.shape == (0, K) and w.shape == (0, K)

    off = torch.full((E + 1,), 7, dtype=torch.int32, device="cuda")
    wsp = moe.workspace("permute", N=0, E=E)
    off, ps, ip, xp = moe.moe_permute(x, ids, E, expert_offsets=off, ws=wsp)
    assert moe.read_device_error(wsp) == moe.MOE_OK
    assert torch.equal(off.cpu(), torch.zeros(E + 1, dtype=torch.int32))

    wsf = moe.workspace("ffn", 0, D, E, 1, Dff)
    h, y = moe.moe_grouped_ffn(xp, off, w1, w3, w2, moe.ACT_SWIGLU, ws=wsf)
    assert h.shape == (0, Dff) and y.shape == (0, D)
    assert moe.read_device_error(wsf) == moe.MOE_OK

    out = moe.moe_combine(y, ip, w)
    assert out.shape == (0, D)

    wsl = moe.workspace("layer", 0, D, E, K, Dff)
    out = moe.moe_layer_forward(x, wg, None, w1, w3, w2, K, 0, moe.ACT_SWIGLU, ws=wsl)
    assert out.shape == (0, D) and moe.read_device_error(wsl) == moe.MOE_OK

    qw = moe.quantize_experts_e4m3(w1, w3, w2)
    ws8 = moe.workspace("layer_e4m3", 0, D, E, K, Dff)
    out = moe.moe_layer_forward_e4m3(x, wg, None, qw, K, 0, moe.ACT_SWIGLU, ws=ws8)
    assert out.shape == (0, D) and moe.read_device_error(ws8) == moe.MOE_OK

    cap = moe.capacity(0, E, K, 1.5)
    assert cap == 0
    wsb = moe.workspace_padded("layer", 0, D, E, K, Dff, cap)
    out = moe.moe_layer_forward_padded(x, wg, None, w1, w3, w2, K, 0, moe.ACT_SWIGLU, cap, ws=wsb)
    assert out.shape == (0, D) and moe.read_device_error(wsb) == moe.MOE_OK
    torch.cuda.synchronize()


@pytest.mark.parametrize("N", [5, 40])
def test_route_at_the_expert_and_k_limits(moe, N):
    # E = 1024 and K = 32, the largest the size checks allow: the CUDA-core
    # logits (5 tokens) and the tensor-core GEMM (40 tokens)
    D, E, K = 128, 1024, 32
    gen = torch.Generator().manual_seed(N)
    x = _bf16((N, D), gen)
    wg = _bf16((E, D), gen, D ** -0.5)
    bias = (torch.randn(E, generator=gen) * 0.5).to(torch.float32)
    for mode in (0, 1):
        L = torch.empty((N, E), dtype=torch.float32, device="cuda")
        ws = moe.workspace("route", N, D, E, K)
        ids, w = moe.moe_route(x.cuda(), wg.cuda(), bias.cuda(), K, mode, logits_out=L, ws=ws)
        assert moe.read_device_error(ws) == moe.MOE_OK
        Lg = L.cpu().numpy().astype(np.float64)
        L64 = O.logits(bits(x), bits(wg), bias.numpy().astype(np.float64))
        assert np.all(np.abs(Lg - L64) <= logits_bound(f64(x), f64(wg), bias.numpy().astype(np.float64)))
        r = O.route_from_logits(Lg, K, mode)
        assert np.array_equal(ids.cpu().numpy(), r["ids"])
        assert np.max(np.abs(w.cpu().numpy() - r["w"])) <= WEIGHT_ATOL
        assert np.allclose(w.cpu().numpy().sum(axis=1), 1.0, atol=1e-5)


@pytest.mark.parametrize("N,K", [(300, 1), (40, 2)])
def test_layer_with_every_token_on_one_expert(moe, N, K):
    # a bias of +50 on expert 3 puts it first for every token: with K = 1 it
    # owns all N rows and every other expert is empty
    from mixture_experts_layer_02_gb300 import synth
    D, E, Dff = 256, 16, 128
    wl = synth.Workload("hot", N, D, E, K, Dff, synth.ACT_SWIGLU, synth.SOFTMAX_TOPK, 0.0)
    inp = synth.make_inputs(wl, seed=N + K)
    bias = torch.zeros(E, dtype=torch.float32)
    bias[3] = 50.0
    dev = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    ws = moe.workspace("layer", N, D, E, K, Dff)
    out = moe.moe_layer_forward(dev["x"], dev["w_gate"], bias.cuda(), dev["w1"], dev["w3"], dev["w2"],
                                K, 0, synth.ACT_SWIGLU, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    mid = moe.layer_intermediates(ws, N, D, E, K, Dff)
    ids = mid["topk_ids"].cpu().numpy()
    assert np.all(ids[:, 0] == 3)
    offs = mid["expert_offsets"].cpu().numpy()
    assert offs[4] - offs[3] == N
    if K == 1:
        assert offs[3] == 0 and offs[E] == N and np.count_nonzero(np.diff(offs)) == 1
    xb = bits(inp["x"])
    full = O.layer(xb, bits(inp["w_gate"]), bias.numpy().astype(np.float64), bits(inp["w1"]), bits(inp["w3"]),
                   bits(inp["w2"]), K, 0, synth.ACT_SWIGLU)
    tie = near_tie_mask(full["logits"], K)
    assert np.array_equal(ids[~tie], full["ids"][~tie])
    assert_close(f64(out)[~tie], full["out"][~tie], "out vs oracle")
