"""Paradigm B (fixed capacity per expert, drops past it) against the oracle:
"MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im), 第二层
范式 B.  Integer outputs (slots, kept counts, offsets, padded rows) are exact;
the layer output uses the layer tolerance."""
import json
import math
import os

import numpy as np
import pytest
import torch

from helpers import WEIGHT_ATOL, assert_close, bits, f64, random_ids
from oracle import oracle as O

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def test_padded_permute_page_example(moe):
    g = json.load(open(os.path.join(GOLDEN, "permutation_example.json")))
    ids = torch.tensor(g["assignment"], dtype=torch.int32).view(-1, 1)
    x = torch.randn((8, 64), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    for cap in (8, 2):
        off, kept, slot, xp = moe.moe_permute_padded(x.cuda(), ids.cuda(), 3, cap)
        o_slot, o_kept = O.place_padded(ids.numpy(), 3, cap)
        assert off.cpu().tolist() == [0, cap, 2 * cap, 3 * cap]
        assert np.array_equal(kept.cpu().numpy(), o_kept)
        assert np.array_equal(slot.cpu().numpy(), o_slot)
        assert np.array_equal(bits(xp), O.padded_rows(bits(x), o_slot, 3, cap))


@pytest.mark.parametrize("N,E,K,D,factor,skew", [
    (300, 16, 4, 128, 1.5, 2.0), (1000, 64, 8, 64, 1.0, 1.2), (40, 8, 2, 64, 0.5, None),
    (4096, 256, 8, 64, 1.5, 1.2), (17, 4, 2, 64, 0.0, None), (64, 8, 2, 128, 4.0, None),
])
def test_padded_permute_matches_oracle(moe, N, E, K, D, factor, skew):
    gen = torch.Generator().manual_seed(N + E)
    ids = random_ids(N, E, K, gen, skew)
    x = torch.randn((N, D), generator=gen).to(torch.bfloat16)
    cap = moe.capacity(N, E, K, factor)
    assert cap == math.ceil(factor * N * K / E - 1e-9)
    ws = moe.workspace_padded("permute", N=N, E=E, cap=cap)
    off, kept, slot, xp = moe.moe_permute_padded(x.cuda(), ids.cuda(), E, cap, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    o_slot, o_kept = O.place_padded(ids.numpy(), E, cap)
    assert np.array_equal(kept.cpu().numpy(), o_kept)
    assert np.array_equal(slot.cpu().numpy(), o_slot)
    assert np.array_equal(off.cpu().numpy(), np.arange(0, E * cap + 1, max(cap, 1))[:E + 1] if cap else np.zeros(E + 1))
    assert np.array_equal(bits(xp), O.padded_rows(bits(x), o_slot, E, cap))


def test_padded_combine_matches_oracle(moe):
    gen = torch.Generator().manual_seed(3)
    N, K, E, cap, D = 200, 4, 16, 30, 256
    y = torch.randn((E * cap, D), generator=gen).to(torch.bfloat16)
    slot = torch.randint(-1, E * cap, (N, K), generator=gen, dtype=torch.int32)
    w = torch.softmax(torch.randn((N, K), generator=gen), -1).to(torch.float32)
    ws = moe.workspace("combine")
    out = moe.moe_combine_padded(y.cuda(), slot.cuda(), w.cuda(), E, cap, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK          # -1 is a drop, not an error
    ref = O.combine_kept(f64(y), slot.numpy(), w.numpy().astype(np.float64))
    S = O.combine_kept(np.abs(f64(y)), slot.numpy(), np.abs(w.numpy().astype(np.float64)))
    assert np.all(np.abs(f64(out) - ref) <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -23 * S + 1e-30)


@pytest.mark.parametrize("N,D,E,K,Dff,act,mode,zipf,factor", [
    (64, 128, 8, 2, 256, 0, 0, 0.0, 1.0),
    (300, 128, 32, 8, 128, 1, 1, 1.2, 1.5),
    (77, 256, 16, 4, 192, 1, 0, 0.0, 0.6),
    (40, 64, 4, 2, 64, 1, 0, 0.0, 0.0),       # capacity 0: everything dropped
])
def test_padded_layer_matches_oracle(moe, N, D, E, K, Dff, act, mode, zipf, factor):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.Workload("p", N, D, E, K, Dff, act, mode, zipf)
    inp = synth.make_inputs(wl, seed=N + K)
    dev = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    cap = moe.capacity(N, E, K, factor)
    ws = moe.workspace_padded("layer", N, D, E, K, Dff, cap)
    out = moe.moe_layer_forward_padded(dev["x"], dev["w_gate"], dev["bias"], dev["w1"], dev["w3"], dev["w2"],
                                       K, mode, act, cap, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    mid = moe.layer_padded_intermediates(ws, N, D, E, K, Dff, cap)
    # routing from the GPU's own logits, then padded placement, exact
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    moe.moe_route(dev["x"], dev["w_gate"], dev["bias"], K, mode, logits_out=L)
    r = O.route_from_logits(L.cpu().numpy().astype(np.float64), K, mode)
    assert np.array_equal(mid["topk_ids"].cpu().numpy(), r["ids"])
    assert np.max(np.abs(mid["topk_w"].cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    slot, kept = O.place_padded(r["ids"], E, cap)
    assert np.array_equal(mid["slot"].cpu().numpy(), slot)
    assert np.array_equal(mid["kept"].cpu().numpy(), kept)
    xp = O.padded_rows(bits(inp["x"]), slot, E, cap)
    assert np.array_equal(bits(mid["x_pad"]), xp)
    # FFN over the padded buffer and the kept-only weighted sum, in fp64
    off = np.arange(0, E * cap + 1, cap, dtype=np.int32) if cap else np.zeros(E + 1, np.int32)
    y = O.grouped_ffn(xp, off, bits(inp["w1"]), None if inp["w3"] is None else bits(inp["w3"]),
                      bits(inp["w2"]), act) if cap else np.zeros((0, D))
    ref = O.combine_kept(y, slot, r["w"])
    if cap == 0:
        assert torch.count_nonzero(out) == 0
    else:
        assert (slot < 0).any() or factor >= 1.0
        assert_close(f64(out), ref, "padded out")
