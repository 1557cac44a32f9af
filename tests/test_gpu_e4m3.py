"""Parity of the FP8 (e4m3) path against the fp64 oracle, through the C ABI.

Quantisation is integer work decided by floating point: the GPU's codes and
scales must equal the oracle's bit for bit, and the oracle's FP8 GEMMs take
the GPU's own quantised inputs stage by stage (h from x and the weights, the
codes of h from the GPU's bf16 h, y from the GPU's codes of h), so each stage
is checked on identical inputs.  The GEMMs multiply exact e4m3 products and
accumulate in fp32, so the bf16 path's tolerances hold unchanged."""
import numpy as np
import pytest
import torch

from helpers import WEIGHT_ATOL, assert_close, bits, f64, near_tie_mask
from oracle import oracle as O
from test_gpu_kernels import FFN_MODES, _graph_kernel_nodes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _no_device_error(moe, ws):
    assert moe.read_device_error(ws) == moe.MOE_OK


def _rows_spread(shape, gen, lo=-8, hi=8, scale=1.0):
    """bf16 rows whose magnitudes differ by powers of two (distinct scales)."""
    t = torch.randn(shape, generator=gen, dtype=torch.float32) * scale
    e = torch.randint(lo, hi + 1, shape[:-1] + (1,), generator=gen).to(torch.float32)
    return (t * torch.pow(2.0, e)).to(torch.bfloat16)


def _u8(t):
    return t.detach().cpu().numpy()


# ------------------------------------------------------------------ quantiser
def _quant_inputs(cols):
    gen = torch.Generator().manual_seed(3 + cols)
    rows = [_rows_spread((40, cols), gen, -30, 30)]
    # zero, -0, subnormal bf16 rows, huge rows
    z = torch.zeros((1, cols), dtype=torch.bfloat16)
    nz = torch.full((1, cols), -0.0, dtype=torch.bfloat16)
    mag = torch.randint(0, 128, (1, cols), generator=gen).numpy().astype(np.uint16)     # subnormal bf16
    sign = (torch.randint(0, 2, (1, cols), generator=gen).numpy().astype(np.uint16) << 15).astype(np.uint16)
    sub = torch.from_numpy((mag | sign).view(np.int16)).view(torch.bfloat16)
    big = (torch.randn((1, cols), generator=gen) * 3e37).to(torch.bfloat16)
    # exact e4m3 ties after scaling: row max 448 fixes the scale at 1
    pat = [448.0, 1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, 1.875 * 2 ** -6 + 2 ** -10,
           -(2.0 ** -11), 0.0, -0.0]
    ties = torch.tensor((pat * (cols // len(pat) + 1))[:cols], dtype=torch.float32)
    rows += [z, nz, sub, big, ties.view(1, -1).to(torch.bfloat16)]
    return torch.cat(rows, 0)


# one CTA per row with 1..8 chunks per thread, and the two-pass path past 16384
@pytest.mark.parametrize("cols", [16, 768, 2048, 4096, 7168, 14336, 16384, 20480])
def test_quantize_matches_oracle_bit_exact(moe, cols):
    x = _quant_inputs(cols)
    q, s = moe.moe_quantize_e4m3(x.cuda())
    oq, os_ = O.quant_rows_e4m3(bits(x))
    assert np.array_equal(_u8(q), oq)
    assert np.array_equal(s.cpu().numpy(), os_)


def test_quantize_weight_stack_shape(moe):
    gen = torch.Generator().manual_seed(4)
    w = _rows_spread((3, 256, 384), gen)
    q, s = moe.moe_quantize_e4m3(w.cuda())
    assert q.shape == (3, 256, 384) and s.shape == (3, 256)
    oq, os_ = O.quant_rows_e4m3(bits(w))
    assert np.array_equal(_u8(q), oq) and np.array_equal(s.cpu().numpy(), os_)


# ------------------------------------------------------------------ grouped FFN
def _ffn8_case(moe, counts, D, Dff, act, seed, indexed):
    gen = torch.Generator().manual_seed(seed)
    E = len(counts)
    rows = int(sum(counts))
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    x = _rows_spread((rows, D), gen)
    w1 = _rows_spread((E, Dff, D), gen, -3, 3, D ** -0.5)
    w3 = _rows_spread((E, Dff, D), gen, -3, 3, D ** -0.5) if act == 1 else None
    w2 = _rows_spread((E, D, Dff), gen, -3, 3, Dff ** -0.5)
    qw = moe.quantize_experts_e4m3(w1.cuda(), None if w3 is None else w3.cuda(), w2.cuda())
    xq, sx = moe.moe_quantize_e4m3(x.cuda())
    # the quantised operands are the oracle's, bit for bit
    o_xq, o_sx = O.quant_rows_e4m3(bits(x))
    o_w1q, o_s1 = O.quant_rows_e4m3(bits(w1))
    o_w2q, o_s2 = O.quant_rows_e4m3(bits(w2))
    assert np.array_equal(_u8(xq), o_xq) and np.array_equal(sx.cpu().numpy(), o_sx)
    assert np.array_equal(_u8(qw["w1q"]), o_w1q) and np.array_equal(qw["s1"].cpu().numpy(), o_s1)
    assert np.array_equal(_u8(qw["w2q"]), o_w2q) and np.array_equal(qw["s2"].cpu().numpy(), o_s2)
    o_w3q = o_s3 = None
    if w3 is not None:
        o_w3q, o_s3 = O.quant_rows_e4m3(bits(w3))
        assert np.array_equal(_u8(qw["w3q"]), o_w3q) and np.array_equal(qw["s3"].cpu().numpy(), o_s3)
    # rows reach the FFN either with their own scales or through an index
    # (as the layer does: token scales read through perm_src)
    if indexed:
        idx = torch.randperm(rows, generator=gen).to(torch.int32)
        xq_perm = xq[idx.cuda().long()].contiguous()
        o_xq_perm, o_sx_perm = o_xq[idx.numpy()], o_sx[idx.numpy()]
        x_scale, x_index = sx, idx.cuda()
    else:
        xq_perm, o_xq_perm, o_sx_perm = xq, o_xq, o_sx
        x_scale, x_index = sx, None
    ws = moe.workspace("ffn", rows, D, E, 1, Dff)
    h, hq, hs, y = moe.moe_grouped_ffn_e4m3(xq_perm, x_scale, x_index, off.cuda(), qw["w1q"], qw["s1"],
                                            qw["w3q"], qw["s3"], qw["w2q"], qw["s2"], act, ws=ws)
    _no_device_error(moe, ws)
    hg = bits(h)
    h_ref = np.zeros((rows, Dff))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if a < b:
            h_ref[a:b] = O.expert_up_e4m3(o_xq_perm[a:b], o_sx_perm[a:b], o_w1q[e], o_s1[e],
                                          None if o_w3q is None else o_w3q[e],
                                          None if o_s3 is None else o_s3[e], act)
    assert_close(O.bf16_to_f64(hg), h_ref, "h")
    assert np.all(np.abs(O.bf16_to_f64(hg) - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 2e-3 * np.abs(h_ref).max())
    # the codes of h: the oracle's quantisation of the GPU's own bf16 h
    r_hq, r_hs = O.quant_rows_e4m3(hg)
    assert np.array_equal(_u8(hq), r_hq) and np.array_equal(hs.cpu().numpy(), r_hs)
    y_ref = np.zeros((rows, D))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if a < b:
            y_ref[a:b] = O.expert_down_e4m3(r_hq[a:b], r_hs[a:b], o_w2q[e], o_s2[e])
    assert_close(f64(y), y_ref, "y_perm")


FFN8_CASES = [
    ([0, 1, 127, 129, 300], 128, 256, 1),
    ([0, 1, 127, 129, 300], 128, 256, 0),
    ([64], 128, 256, 0),
    ([5, 0, 0, 260, 3], 256, 128, 1),
    ([1, 2, 3, 4, 5, 6, 7, 8], 512, 768, 1),
    ([200, 0, 57, 384], 256, 128, 1),
    ([3, 5], 2048, 1024, 1),       # few tiles: split-K of both GEMMs
    ([3, 5], 2048, 1024, 0),
]


@pytest.mark.parametrize("counts,D,Dff,act", FFN8_CASES)
@pytest.mark.parametrize("mode", list(FFN_MODES))
def test_grouped_ffn_e4m3_matches_oracle(moe, counts, D, Dff, act, mode, monkeypatch):
    for k, v in FFN_MODES[mode].items():
        monkeypatch.setenv(k, v)
    _ffn8_case(moe, counts, D, Dff, act, seed=len(counts) * 31 + D + Dff + act, indexed=(mode == "auto"))


@pytest.mark.parametrize("counts,D,Dff,act", [
    ([300, 0, 513, 1, 256], 256, 256, 1),
    ([700, 900, 3, 258], 512, 1024, 1),
    ([512, 0, 100], 512, 256, 0),
])
def test_grouped_ffn_e4m3_on_cta_pairs_matches_oracle(moe, counts, D, Dff, act, monkeypatch):
    monkeypatch.setenv("MOE_PAIR_GEMM", "1")
    _ffn8_case(moe, counts, D, Dff, act, seed=11 * len(counts) + D + Dff + act, indexed=True)


def test_e4m3_rejects_widths_not_multiple_of_128(moe):
    xq = torch.zeros((4, 192), dtype=torch.uint8).cuda()
    sx = torch.ones(4).cuda()
    off = torch.tensor([0, 4], dtype=torch.int32).cuda()
    w = torch.zeros((1, 128, 192), dtype=torch.uint8).cuda()
    s = torch.ones((1, 128)).cuda()
    w2 = torch.zeros((1, 192, 128), dtype=torch.uint8).cuda()
    s2 = torch.ones((1, 192)).cuda()
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_grouped_ffn_e4m3(xq, sx, None, off, w, s, w, s, w2, s2, 1)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


# ------------------------------------------------------------------ whole layer
@pytest.mark.parametrize("N,D,E,K,Dff,act,mode,zipf", [
    (64, 128, 8, 2, 256, 0, 0, 0.0),          # the tiny workload
    (1, 128, 8, 2, 256, 1, 0, 0.0),
    (77, 256, 16, 4, 256, 1, 1, 0.0),
    (300, 128, 32, 8, 128, 1, 1, 1.2),
    (130, 128, 1, 1, 128, 1, 0, 0.0),
    (2048, 256, 4, 2, 256, 1, 0, 0.0),        # enough rows per expert for CTA pairs
])
def test_layer_e4m3_matches_oracle(moe, N, D, E, K, Dff, act, mode, zipf):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.Workload("t", N, D, E, K, Dff, act, mode, zipf)
    inp = synth.make_inputs(wl, seed=N + E + 1)
    dev = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    qw = moe.quantize_experts_e4m3(dev["w1"], dev["w3"], dev["w2"])
    ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
    out = moe.moe_layer_forward_e4m3(dev["x"], dev["w_gate"], dev["bias"], qw, K, mode, act, ws=ws)
    _no_device_error(moe, ws)
    mid = moe.layer_e4m3_intermediates(ws, N, D, E, K, Dff)
    # routing: the bf16 router, checked as in the bf16 layer
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids2, _ = moe.moe_route(dev["x"], dev["w_gate"], dev["bias"], K, mode, logits_out=L)
    assert torch.equal(ids2, mid["topk_ids"])
    r = O.route_from_logits(L.cpu().numpy().astype(np.float64), K, mode)
    assert np.array_equal(mid["topk_ids"].cpu().numpy(), r["ids"])
    assert np.max(np.abs(mid["topk_w"].cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    assert np.array_equal(mid["expert_offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(mid["perm_src"].cpu().numpy(), r["perm_src"])
    # tokens quantised once, codes moved by the permutation: exact
    xb = bits(inp["x"])
    o_xq, o_sx = O.quant_rows_e4m3(xb)
    assert np.array_equal(_u8(mid["xq"]), o_xq) and np.array_equal(mid["x_scale"].cpu().numpy(), o_sx)
    assert np.array_equal(_u8(mid["xq_perm"]), o_xq[r["perm_src"]])
    # FFN stages on the GPU's routing
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
    # and the oracle's whole FP8 chain from its own fp64 logits
    b64 = None if inp["bias"] is None else inp["bias"].numpy().astype(np.float64)
    full = O.layer_e4m3(xb, bits(inp["w_gate"]), b64, o_w1q, o_s1, o_w3q, o_s3, o_w2q, o_s2, K, mode, act)
    tie = near_tie_mask(full["logits"], K)
    assert_close(f64(out)[~tie], full["out"][~tie], "out vs full oracle")


@pytest.mark.parametrize("N,D,E,K,Dff", [(64, 128, 8, 2, 256), (4, 2048, 128, 8, 768), (700, 256, 16, 8, 128)])
def test_layer_e4m3_launch_count_is_what_runs(moe, N, D, E, K, Dff):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.Workload("c", N, D, E, K, Dff, 1, 0, 0.0)
    inp = {k: (None if v is None else v.cuda()) for k, v in synth.make_inputs(wl, seed=2).items()}
    qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
    ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
    run = lambda: moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], None, qw, K, 0, 1, ws=ws)
    run()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(gr):
        run()
    assert _graph_kernel_nodes(gr.raw_cuda_graph()) == moe.layer_launches_e4m3(N, D, E, K, Dff, 1)
