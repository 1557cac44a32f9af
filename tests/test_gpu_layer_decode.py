"""The one-launch decode layer (layer_decode.cu): a layer call of up to 8
tokens runs router logits, top-K, placement, GEMM1 + activation, GEMM2 and
the combine in one cooperative launch.

Checked against the fp64 oracle like the chain of launches: routing and
permutation exact (and bit-identical to the chain's, which uses the same
routing functions), h / y_perm per expert and the output within the bf16
tolerance; plus launch accounting, graph replay, repeated calls on one
workspace (the grid barrier's words persist in its header), a withheld
barrier arrival that must time out without hanging, and NaN tokens.
"""
import time

import numpy as np
import pytest
import torch

from helpers import WEIGHT_ATOL, assert_close, bits, f64, near_tie_mask
from oracle import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _inputs(N, D, E, K, Dff, act, mode, zipf=0.0, seed=0):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.Workload("d", N, D, E, K, Dff, act, mode, zipf)
    inp = synth.make_inputs(wl, seed=seed)
    return {k: (None if v is None else v.cuda()) for k, v in inp.items()}


def _layer(moe, inp, K, mode, act, ws=None):
    return moe.moe_layer_forward(inp["x"], inp["w_gate"], inp["bias"], inp["w1"], inp["w3"], inp["w2"],
                                 K, mode, act, ws=ws)


# N, D, E, K, Dff, act, mode: token counts 1..8 (each rows-per-expert
# instantiation), D with a partial last chunk batch (192, 7168), D_ffn over
# several GEMM2 batches (2048), E up to 256, K up to 32 with N*K = 64, one
# expert, both activations and both score functions.
SHAPES = [
    (1, 2048, 128, 8, 768, 1, 0),      # Qwen3-shaped, one token
    (1, 256, 16, 4, 128, 0, 1),        # SiLU
    (2, 128, 8, 2, 256, 1, 1),
    (3, 192, 20, 5, 64, 1, 0),
    (4, 128, 256, 16, 64, 1, 1),       # E = 256, 64 rows
    (5, 64, 1, 1, 64, 1, 0),           # one expert
    (8, 512, 64, 8, 128, 0, 1),        # 64 rows, SiLU
    (2, 256, 64, 32, 64, 1, 0),        # K = 32
    (2, 7168, 16, 4, 128, 1, 1),       # long rows: several GEMM1 chunk batches
    (1, 256, 8, 2, 2048, 1, 0),        # long D_ffn: several GEMM2 chunk batches
    (7, 1024, 32, 4, 256, 1, 1),
]


@pytest.mark.parametrize("w2smem", ["0", "1"])
@pytest.mark.parametrize("N,D,E,K,Dff,act,mode", SHAPES)
def test_decode_layer_matches_oracle(moe, N, D, E, K, Dff, act, mode, w2smem, monkeypatch):
    """Every intermediate against the oracle, with GEMM2 reading W2 from
    global memory (the default) and, where the CTAs' W2 rows fit, from the
    copy staged in shared memory (MOE_LAYER_DECODE_W2_SMEM=1)."""
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    monkeypatch.setenv("MOE_LAYER_DECODE_W2_SMEM", w2smem)
    assert moe.layer_launches(N, D, E, K, Dff, act) == 1
    # the DeepSeek-style score (mode 1) with the Zipf-shaped router bias
    inp = _inputs(N, D, E, K, Dff, act, mode, zipf=1.2 if mode == 1 else 0.0, seed=N * 31 + E)
    assert (inp["bias"] is not None) == (mode == 1)
    ws = moe.workspace("layer", N, D, E, K, Dff)
    out = _layer(moe, inp, K, mode, act, ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    mid = moe.layer_intermediates(ws, N, D, E, K, Dff)

    # routing: the same bits as moe_route, and the oracle's selection from those logits
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids2, w2 = moe.moe_route(inp["x"], inp["w_gate"], inp["bias"], K, mode, logits_out=L)
    assert torch.equal(ids2, mid["topk_ids"]) and torch.equal(w2, mid["topk_w"])
    r = O.route_from_logits(L.cpu().numpy().astype(np.float64), K, mode)
    assert np.array_equal(mid["topk_ids"].cpu().numpy(), r["ids"])
    assert np.max(np.abs(mid["topk_w"].cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    assert np.array_equal(mid["expert_offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(mid["perm_src"].cpu().numpy(), r["perm_src"])
    assert np.array_equal(mid["inv_perm"].cpu().numpy(), r["inv_perm"])
    xb = bits(inp["x"])
    assert np.array_equal(bits(mid["x_perm"]), O.gather_rows(xb, r["perm_src"]))

    # h and y_perm, expert by expert: h from x_perm, y from the GPU's own bf16 h
    off = r["offsets"]
    xp = bits(mid["x_perm"])
    h_gpu, y_gpu = bits(mid["h"]), bits(mid["y_perm"])
    h_ref = np.empty((N * K, Dff))
    y_ref = np.empty((N * K, D))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        w3e = None if inp["w3"] is None else bits(inp["w3"][e])
        h_ref[a:b] = O.expert_up(xp[a:b], bits(inp["w1"][e]), w3e, act)
        y_ref[a:b] = O.expert_down(h_gpu[a:b], bits(inp["w2"][e]))
    assert_close(O.bf16_to_f64(h_gpu), h_ref, "h")
    assert_close(O.bf16_to_f64(y_gpu), y_ref, "y_perm")

    # the combine of the GPU's y_perm: the oracle's weighted sum in k order
    ref_c = O.combine(O.bf16_to_f64(y_gpu), r["inv_perm"], r["w"])
    assert_close(f64(out), ref_c, "out from y_perm")
    # and the whole fp64 chain from x
    b64 = None if inp["bias"] is None else inp["bias"].cpu().numpy().astype(np.float64)
    full = O.layer(xb, bits(inp["w_gate"]), b64, bits(inp["w1"]), None if inp["w3"] is None else bits(inp["w3"]),
                   bits(inp["w2"]), K, mode, act)
    tie = near_tie_mask(full["logits"], K)
    assert_close(f64(out)[~tie], full["out"][~tie], "out vs fp64 chain")


@pytest.mark.parametrize("N,D,E,K,Dff,act,mode", [SHAPES[0], SHAPES[4], SHAPES[6]])
def test_decode_layer_agrees_with_the_chain_of_launches(moe, N, D, E, K, Dff, act, mode, monkeypatch):
    """Routing, placement and x_perm are bit-identical to the separate
    kernels'; h, y_perm and the output agree within the bf16 tolerance (the
    GEMM sums run in another order)."""
    inp = _inputs(N, D, E, K, Dff, act, mode, seed=7)
    res = {}
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    for flag in ("1", "0"):
        monkeypatch.setenv("MOE_LAYER_DECODE", flag)
        ws = moe.workspace("layer", N, D, E, K, Dff)
        out = _layer(moe, inp, K, mode, act, ws)
        assert moe.read_device_error(ws) == moe.MOE_OK
        res[flag] = (out, moe.layer_intermediates(ws, N, D, E, K, Dff))
    assert moe.layer_launches(N, D, E, K, Dff, act) > 1   # MOE_LAYER_DECODE=0: the chain
    (o1, m1), (o0, m0) = res["1"], res["0"]
    for k in ("topk_ids", "topk_w", "expert_offsets", "perm_src", "inv_perm", "x_perm"):
        assert torch.equal(m1[k], m0[k]), k
    assert_close(f64(m1["h"]), f64(m0["h"]), "h")
    assert_close(f64(m1["y_perm"]), f64(m0["y_perm"]), "y_perm")
    assert_close(f64(o1), f64(o0), "out")


def test_decode_layer_repeated_calls_and_graph_replay(moe, monkeypatch):
    """Many calls on one workspace (the barrier words persist in its header)
    and graph replays give the same bits every time; the graph holds one
    kernel node."""
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    N, D, E, K, Dff = 1, 2048, 128, 8, 768
    inp = _inputs(N, D, E, K, Dff, 1, 0, seed=3)
    ws = moe.workspace("layer", N, D, E, K, Dff)
    out = torch.empty((N, D), dtype=torch.bfloat16, device="cuda")
    ref = _layer(moe, inp, K, 0, 1, ws).clone()
    for _ in range(40):
        moe.moe_layer_forward(inp["x"], inp["w_gate"], inp["bias"], inp["w1"], inp["w3"], inp["w2"], K, 0, 1,
                              out=out, ws=ws)
        assert torch.equal(out, ref)
    assert moe.read_device_error(ws) == moe.MOE_OK
    out.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g):
        moe.moe_layer_forward(inp["x"], inp["w_gate"], inp["bias"], inp["w1"], inp["w3"], inp["w2"], K, 0, 1,
                              out=out, ws=ws)
    from test_gpu_kernels import _graph_kernel_nodes
    assert _graph_kernel_nodes(g.raw_cuda_graph()) == 1
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert moe.read_device_error(ws) == moe.MOE_OK


def test_decode_layer_withheld_arrival_times_out(moe, monkeypatch):
    """Debug bit 0 makes CTA 0 leave before its first grid-barrier arrival:
    every other CTA's bounded wait runs out, the call reports
    MOE_ERR_DEVICE_TIMEOUT, and after the header is cleared the context and
    the workspace compute correctly again."""
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    N, D, E, K, Dff = 2, 256, 16, 4, 128
    inp = _inputs(N, D, E, K, Dff, 1, 1, seed=11)
    ws = moe.workspace("layer", N, D, E, K, Dff)
    ref = _layer(moe, inp, K, 1, 1, ws).clone()
    assert moe.read_device_error(ws) == moe.MOE_OK
    moe.set_debug_flags(ws, 1)
    t0 = time.time()
    _layer(moe, inp, K, 1, 1, ws)
    status = moe.read_device_error(ws)
    assert status == moe.MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30.0
    moe.clear_device_error(ws)
    out = _layer(moe, inp, K, 1, 1, ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(out, ref)


def test_decode_layer_nan_token(moe, monkeypatch):
    """A token whose logits are NaN gets no expert: the call records
    MOE_ERR_DEVICE_BOUNDS, its output row is zero, and the other tokens are
    what the chain of launches gives them."""
    N, D, E, K, Dff = 3, 256, 16, 4, 128
    inp = _inputs(N, D, E, K, Dff, 1, 0, seed=5)
    inp["x"][1, 7] = float("nan")
    outs = {}
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    for flag in ("1", "0"):
        monkeypatch.setenv("MOE_LAYER_DECODE", flag)
        ws = moe.workspace("layer", N, D, E, K, Dff)
        outs[flag] = _layer(moe, inp, K, 0, 1, ws)
        assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_BOUNDS
        mid = moe.layer_intermediates(ws, N, D, E, K, Dff)
        assert torch.all(mid["topk_ids"][1] == -1) and torch.all(mid["inv_perm"][1] == -1)
        assert int(mid["expert_offsets"][E]) == (N - 1) * K
    assert torch.all(outs["1"][1] == 0)
    keep = torch.tensor([0, 2], device="cuda")
    assert_close(f64(outs["1"][keep]), f64(outs["0"][keep]), "valid tokens")


@pytest.mark.parametrize("N,K", [(9, 4), (4, 20)])
def test_decode_layer_limits(moe, N, K, monkeypatch):
    """Beyond 8 tokens or 64 assignments the layer runs the chain of launches."""
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    assert moe.layer_launches(N, 256, 64, K, 128, 1) > 1


def test_decode_layer_default_token_limit(moe, monkeypatch):
    """Without the tuning variables the layer runs as one launch for the
    token counts where that measured faster on GB300 (Qwen3-shaped layer: up
    to 4 tokens with bf16 or e4m3 experts) and as the chain of launches
    above."""
    monkeypatch.delenv("MOE_LAYER_DECODE", raising=False)
    monkeypatch.delenv("MOE_LAYER_DECODE_MAX_N", raising=False)
    for n in (1, 2, 3, 4):
        assert moe.layer_launches(n, 2048, 128, 8, 768, 1) == 1
    assert moe.layer_launches(5, 2048, 128, 8, 768, 1) > 1
    for n in (1, 2, 3, 4):
        assert moe.layer_launches_e4m3(n, 2048, 128, 8, 768, 1) == 1
    assert moe.layer_launches_e4m3(5, 2048, 128, 8, 768, 1) > 1
    monkeypatch.setenv("MOE_LAYER_DECODE", "0")
    assert moe.layer_launches(1, 2048, 128, 8, 768, 1) > 1
    assert moe.layer_launches_e4m3(1, 2048, 128, 8, 768, 1) > 1


# ------------------------------------------------------------------ e4m3 experts
def _u8(t):
    return t.detach().contiguous().cpu().numpy().astype(np.uint8)


# N, D, E, K, Dff, act, mode, W2 staged in shared memory (1) or read from
# global memory (0): one to eight tokens, SwiGLU and SiLU, both score functions
E4M3_SHAPES = [
    (1, 2048, 128, 8, 768, 1, 0, "1"),      # Qwen3-shaped, one token
    (1, 2048, 128, 8, 768, 1, 0, "0"),      # the same with W2 from global memory
    (2, 2048, 128, 8, 768, 1, 1, "1"),      # two tokens: 16 expert slots
    (1, 256, 16, 4, 128, 0, 1, "1"),        # SiLU
    (2, 512, 64, 8, 256, 1, 0, "1"),
    (4, 2048, 128, 8, 768, 1, 1, "1"),      # 32 slots: W2 does not fit, read from global memory
    (3, 1024, 32, 4, 384, 1, 0, "1"),       # 4-column B operand with 3 token rows
    (8, 512, 64, 8, 256, 0, 0, "1"),        # 64 rows, SiLU
    (1, 7168, 16, 4, 256, 1, 1, "1"),       # 48 columns per CTA: three W2 tiles per slot
]


@pytest.mark.parametrize("N,D,E,K,Dff,act,mode,w2smem", E4M3_SHAPES)
def test_decode_layer_e4m3_matches_oracle(moe, N, D, E, K, Dff, act, mode, w2smem, monkeypatch):
    """e4m3 experts in the one launch: the tokens and h quantised by the row
    quantiser's rule (codes and scales bit-exact against the oracle's), both
    GEMMs on the tensor cores over the codes (W2 staged in shared memory or
    read from global memory), every intermediate of the e4m3 layer written."""
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    monkeypatch.setenv("MOE_LAYER_DECODE_W2_SMEM", w2smem)
    assert moe.layer_launches_e4m3(N, D, E, K, Dff, act) == 1
    inp = _inputs(N, D, E, K, Dff, act, mode, zipf=1.2 if mode == 1 else 0.0, seed=N * 17 + E)
    qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
    ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
    out = moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], inp["bias"], qw, K, mode, act, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    mid = moe.layer_e4m3_intermediates(ws, N, D, E, K, Dff)
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids2, w2g = moe.moe_route(inp["x"], inp["w_gate"], inp["bias"], K, mode, logits_out=L)
    assert torch.equal(ids2, mid["topk_ids"]) and torch.equal(w2g, mid["topk_w"])
    r = O.route_from_logits(L.cpu().numpy().astype(np.float64), K, mode)
    assert np.array_equal(mid["expert_offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(mid["perm_src"].cpu().numpy(), r["perm_src"])
    assert np.array_equal(mid["inv_perm"].cpu().numpy(), r["inv_perm"])
    xb = bits(inp["x"])
    o_xq, o_sx = O.quant_rows_e4m3(xb)
    assert np.array_equal(_u8(mid["xq"]), o_xq) and np.array_equal(mid["x_scale"].cpu().numpy(), o_sx)
    assert np.array_equal(_u8(mid["xq_perm"]), o_xq[r["perm_src"]])
    o_w1q, o_s1 = O.quant_rows_e4m3(bits(inp["w1"]))
    o_w2q, o_s2 = O.quant_rows_e4m3(bits(inp["w2"]))
    o_w3q, o_s3 = O.quant_rows_e4m3(bits(inp["w3"])) if inp["w3"] is not None else (None, None)
    g = O.grouped_ffn_e4m3(o_xq[r["perm_src"]], o_sx[r["perm_src"]], r["offsets"], o_w1q, o_s1, o_w3q, o_s3,
                           o_w2q, o_s2, act)
    assert_close(f64(mid["h"]), g["h"], "h")
    r_hq, r_hs = O.quant_rows_e4m3(bits(mid["h"]))
    assert np.array_equal(_u8(mid["hq"]), r_hq) and np.array_equal(mid["h_scale"].cpu().numpy(), r_hs)
    y_ref = np.zeros((N * K, D))
    for e in range(E):
        a, b = int(r["offsets"][e]), int(r["offsets"][e + 1])
        if a < b:
            y_ref[a:b] = O.expert_down_e4m3(r_hq[a:b], r_hs[a:b], o_w2q[e], o_s2[e])
    assert_close(f64(mid["y_perm"]), y_ref, "y_perm")
    assert_close(f64(out), O.combine(y_ref, r["inv_perm"], r["w"]), "out")
    b64 = None if inp["bias"] is None else inp["bias"].cpu().numpy().astype(np.float64)
    full = O.layer_e4m3(xb, bits(inp["w_gate"]), b64, o_w1q, o_s1, o_w3q, o_s3, o_w2q, o_s2, K, mode, act)
    tie = near_tie_mask(full["logits"], K)
    assert_close(f64(out)[~tie], full["out"][~tie], "out vs the fp64 e4m3 chain")


def test_decode_layer_e4m3_agrees_with_the_chain_and_replays(moe, monkeypatch):
    """Routing, the token codes and their permutation are bit-identical to
    the chain of launches'; the output agrees within the tolerance; graph
    replays repeat the bits."""
    N, D, E, K, Dff = 1, 2048, 128, 8, 768
    inp = _inputs(N, D, E, K, Dff, 1, 0, seed=9)
    qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
    res = {}
    for flag in ("1", "0"):
        monkeypatch.setenv("MOE_LAYER_DECODE", flag)
        ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
        out = moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], None, qw, K, 0, 1, ws=ws)
        assert moe.read_device_error(ws) == moe.MOE_OK
        res[flag] = (out, moe.layer_e4m3_intermediates(ws, N, D, E, K, Dff), ws)
    assert moe.layer_launches_e4m3(N, D, E, K, Dff, 1) > 1   # MOE_LAYER_DECODE=0: the chain
    (o1, m1, ws1), (o0, m0, _) = res["1"], res["0"]
    for k in ("topk_ids", "topk_w", "expert_offsets", "perm_src", "inv_perm", "xq", "x_scale", "xq_perm"):
        assert torch.equal(m1[k], m0[k]), k
    assert_close(f64(o1), f64(o0), "out")
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    ref = o1.clone()
    out = torch.empty_like(ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], None, qw, K, 0, 1, out=out, ws=ws1)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert moe.read_device_error(ws1) == moe.MOE_OK


def _layer_e4m3(moe, inp, qw, K, mode, act, ws):
    return moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], inp["bias"], qw, K, mode, act, ws=ws)


def test_decode_layer_e4m3_withheld_arrival_times_out(moe, monkeypatch):
    """The e4m3 kernel's grid barriers: with CTA 0 leaving before its first
    arrival the call reports MOE_ERR_DEVICE_TIMEOUT within the wait bound, and
    after the header is cleared the workspace gives the same bits as before."""
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    N, D, E, K, Dff = 2, 256, 16, 4, 128
    inp = _inputs(N, D, E, K, Dff, 1, 1, seed=13)
    qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
    assert moe.layer_launches_e4m3(N, D, E, K, Dff, 1) == 1
    ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
    ref = _layer_e4m3(moe, inp, qw, K, 1, 1, ws).clone()
    assert moe.read_device_error(ws) == moe.MOE_OK
    moe.set_debug_flags(ws, 1)
    t0 = time.time()
    _layer_e4m3(moe, inp, qw, K, 1, 1, ws)
    assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 30.0
    moe.clear_device_error(ws)
    out = _layer_e4m3(moe, inp, qw, K, 1, 1, ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(out, ref)


def test_decode_layer_e4m3_nan_token(moe, monkeypatch):
    """e4m3 experts, a token whose logits are NaN: both the one launch and the
    chain record MOE_ERR_DEVICE_BOUNDS and give it no expert; the token codes
    and scales of every token (the NaN one included) are the same bits on both
    paths, its output row is zero, and the other tokens agree."""
    N, D, E, K, Dff = 3, 256, 16, 4, 128
    inp = _inputs(N, D, E, K, Dff, 1, 0, seed=7)
    inp["x"][1, 9] = float("nan")
    qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
    outs, mids = {}, {}
    monkeypatch.setenv("MOE_LAYER_DECODE_MAX_N", "8")
    for flag in ("1", "0"):
        monkeypatch.setenv("MOE_LAYER_DECODE", flag)
        assert (moe.layer_launches_e4m3(N, D, E, K, Dff, 1) == 1) == (flag == "1")
        ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
        outs[flag] = _layer_e4m3(moe, inp, qw, K, 0, 1, ws)
        assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_BOUNDS
        mids[flag] = moe.layer_e4m3_intermediates(ws, N, D, E, K, Dff)
        assert torch.all(mids[flag]["topk_ids"][1] == -1) and torch.all(mids[flag]["inv_perm"][1] == -1)
        assert int(mids[flag]["expert_offsets"][E]) == (N - 1) * K
    for k in ("topk_ids", "expert_offsets", "perm_src", "inv_perm", "xq"):
        assert torch.equal(mids["1"][k], mids["0"][k]), k
    assert torch.equal(mids["1"]["x_scale"].view(torch.int32), mids["0"]["x_scale"].view(torch.int32))
    assert torch.all(outs["1"][1] == 0)
    keep = torch.tensor([0, 2], device="cuda")
    assert_close(f64(outs["1"][keep]), f64(outs["0"][keep]), "valid tokens")


def _shifted(t):
    """A copy of t whose base is 16 bytes past a 32-byte boundary."""
    pad = 16 // t.element_size()
    buf = torch.empty(t.numel() + pad, dtype=t.dtype, device=t.device)
    moved = buf[pad:].view_as(t)
    moved.copy_(t)
    assert moved.data_ptr() % 32 == 16
    return moved


@pytest.mark.parametrize("which", ["w1", "w3", "w2", "w1q", "w2q"])
def test_decode_layer_weights_off_32_byte_boundary_run_the_chain(moe, which, monkeypatch):
    """The one launch reads weights in 32-byte pieces: a weight tensor whose
    base is on a 16-byte but not a 32-byte boundary makes the call run the
    chain of launches (more than one kernel in a captured graph), with the
    result of the aligned copy."""
    from test_gpu_kernels import _graph_kernel_nodes
    monkeypatch.setenv("MOE_LAYER_DECODE", "1")
    N, D, E, K, Dff = 1, 256, 16, 4, 128
    inp = _inputs(N, D, E, K, Dff, 1, 0, seed=21)
    e4m3 = which.endswith("q")
    if e4m3:
        qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
        ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
        run = lambda q: moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], inp["bias"], q, K, 0, 1, out=out, ws=ws)
        args_ok, args_moved = qw, dict(qw, **{which: _shifted(qw[which])})
    else:
        ws = moe.workspace("layer", N, D, E, K, Dff)
        run = lambda w: moe.moe_layer_forward(inp["x"], inp["w_gate"], inp["bias"], w["w1"], w["w3"], w["w2"], K, 0,
                                              1, out=out, ws=ws)
        args_ok = {k: inp[k] for k in ("w1", "w3", "w2")}
        args_moved = dict(args_ok, **{which: _shifted(inp[which])})
    out = torch.empty((N, D), dtype=torch.bfloat16, device="cuda")
    run(args_ok)
    ref = out.clone()
    run(args_moved)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert_close(f64(out), f64(ref), "out")
    torch.cuda.synchronize()
    for args, one in ((args_ok, True), (args_moved, False)):
        g = torch.cuda.CUDAGraph(keep_graph=True)
        with torch.cuda.graph(g):
            run(args)
        assert (_graph_kernel_nodes(g.raw_cuda_graph()) == 1) == one
