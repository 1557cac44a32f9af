"""Per-kernel parity of the CUDA path against the fp64 oracle, through the
C ABI, on small seeded inputs that span several tiles, ragged tails, empty
experts and the degenerate cases (K = 1, E = 1, N = 1)."""
import json
import os

import numpy as np
import pytest
import torch

from helpers import (WEIGHT_ATOL, assert_close, bits, f64, logits_bound, near_tie_mask,
                     random_ids)
from oracle import oracle as O

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * scale).to(torch.bfloat16)


def _no_device_error(moe, ws):
    assert moe.read_device_error(ws) == moe.MOE_OK


# ------------------------------------------------------------------ permute
def test_permute_page_example(moe):
    g = json.load(open(os.path.join(GOLDEN, "permutation_example.json")))
    E, K = g["num_experts"], g["top_k"]
    ids = torch.tensor(g["assignment"], dtype=torch.int32).view(-1, K)
    N = ids.shape[0]
    gen = torch.Generator().manual_seed(0)
    x = _bf16((N, 64), gen)
    ws = moe.workspace("permute", N=N, E=E)
    off, ps, ip, xp = moe.moe_permute(x.cuda(), ids.cuda(), E, ws=ws)
    assert off.cpu().tolist() == g["expert_offsets"]
    assert ps.cpu().tolist() == [t for seg in g["segments"] for t in seg]
    assert torch.equal(xp.cpu(), x[ps.cpu().long()])
    assert ip.cpu().view(-1).tolist() == np.argsort([t for seg in g["segments"] for t in seg]).tolist()
    _no_device_error(moe, ws)


@pytest.mark.parametrize("N,E,K,D,skew", [
    (1, 8, 2, 64, None), (17, 8, 2, 128, None), (64, 8, 2, 128, None), (100, 128, 8, 64, None),
    (333, 5, 3, 192, None), (1000, 256, 8, 64, 1.2), (4096, 256, 8, 64, None), (50, 3, 1, 64, None),
    (40, 1, 1, 64, None), (300, 64, 6, 256, 3.0),
    (2000, 16, 4, 2048, None),     # few token blocks, wide rows: the row copy split in column slices
    (3000, 32, 2, 1152, 1.5),      # two slices of 72 chunks
])
def test_permute_matches_oracle(moe, N, E, K, D, skew):
    gen = torch.Generator().manual_seed(N * 7 + E)
    ids = random_ids(N, E, K, gen, skew)
    x = _bf16((N, D), gen)
    ws = moe.workspace("permute", N=N, E=E)
    off, ps, ip, xp = moe.moe_permute(x.cuda(), ids.cuda(), E, ws=ws)
    o_off = O.offsets(ids.numpy(), E)
    o_ps, o_ip = O.place(ids.numpy(), o_off, E)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(ps.cpu().numpy(), o_ps)
    assert np.array_equal(ip.cpu().numpy(), o_ip)
    assert np.array_equal(bits(xp), O.gather_rows(bits(x), o_ps))
    _no_device_error(moe, ws)


def test_permute_flags_bad_ids(moe):
    ids = torch.tensor([[0, 1], [2, 9], [1, 2]], dtype=torch.int32)   # 9 is outside 0..E-1
    x = torch.zeros((3, 64), dtype=torch.bfloat16)
    ws = moe.workspace("permute", N=3, E=3)
    moe.moe_permute(x.cuda(), ids.cuda(), 3, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_BOUNDS
    moe.clear_device_error(ws)
    assert moe.read_device_error(ws) == moe.MOE_OK


def test_permute_is_deterministic(moe):
    gen = torch.Generator().manual_seed(5)
    ids = random_ids(2000, 64, 4, gen).cuda()
    x = _bf16((2000, 128), gen).cuda()
    a = moe.moe_permute(x, ids, 64)
    b = moe.moe_permute(x, ids, 64)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("N,K,D", [(1, 8, 2048), (7, 1, 64), (64, 2, 128), (333, 3, 192), (2048, 8, 256)])
def test_combine_matches_oracle(moe, N, K, D):
    gen = torch.Generator().manual_seed(N + K)
    y = _bf16((N * K, D), gen)
    inv = torch.randperm(N * K, generator=gen).to(torch.int32).view(N, K)
    w = torch.softmax(torch.randn((N, K), generator=gen), -1).to(torch.float32)
    ws = moe.workspace("combine")
    out = moe.moe_combine(y.cuda(), inv.cuda(), w.cuda(), ws=ws)
    ref = O.combine(f64(y), inv.numpy(), w.numpy().astype(np.float64))
    got = f64(out)
    # one bf16 rounding (2^-9 relative) on top of a K-term fp32 sum
    S = O.combine(np.abs(f64(y)), inv.numpy(), np.abs(w.numpy().astype(np.float64)))
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -23 * S + 1e-30)
    _no_device_error(moe, ws)


def test_combine_flags_bad_rows(moe):
    y = torch.ones((4, 64), dtype=torch.bfloat16).cuda()
    inv = torch.tensor([[0, 1], [2, 7]], dtype=torch.int32).cuda()   # 7 >= N*K
    w = torch.full((2, 2), 0.5).cuda()
    ws = moe.workspace("combine")
    out = moe.moe_combine(y, inv, w, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_BOUNDS
    assert torch.all(out[0] == 1.0) and torch.all(out[1] == 0.5)


# ------------------------------------------------------------------ route
@pytest.mark.parametrize("N,D,E,K,mode,with_bias", [
    (64, 128, 8, 2, 0, False), (300, 256, 128, 8, 0, False), (1000, 512, 256, 8, 1, True),
    (129, 64, 3, 1, 0, False), (5, 64, 256, 8, 1, False), (257, 192, 60, 6, 1, True),
    (130, 128, 1, 1, 0, False), (200, 64, 33, 32, 0, True),
    # up to 32 tokens the logits come from the CUDA-core kernel (one warp per expert)
    (1, 2048, 128, 8, 0, False), (8, 2048, 128, 8, 0, True), (17, 512, 60, 6, 1, True),
    (32, 7168, 256, 8, 1, True), (32, 4096, 8, 2, 0, False), (33, 2048, 128, 8, 0, False),
])
def test_route_matches_oracle(moe, N, D, E, K, mode, with_bias):
    gen = torch.Generator().manual_seed(N * 3 + E)
    x = _bf16((N, D), gen)
    wg = _bf16((E, D), gen, D ** -0.5)
    bias = (torch.randn(E, generator=gen) * 2).to(torch.float32) if with_bias else None
    ws = moe.workspace("route", N, D, E, K)
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids, w = moe.moe_route(x.cuda(), wg.cuda(), None if bias is None else bias.cuda(), K, mode,
                           logits_out=L, ws=ws)
    _no_device_error(moe, ws)
    Lg = L.cpu().numpy().astype(np.float64)
    # fp32 logits against the fp64 definition
    b64 = None if bias is None else bias.numpy().astype(np.float64)
    L64 = O.logits(bits(x), bits(wg), b64)
    assert np.all(np.abs(Lg - L64) <= logits_bound(f64(x), f64(wg), b64))
    # given identical fp32 logits: ids bit-exact, weights within 2e-6
    r = O.route_from_logits(Lg, K, mode)
    assert np.array_equal(ids.cpu().numpy(), r["ids"])
    assert np.max(np.abs(w.cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    # against the oracle's own fp64 logits, near-ties excluded and counted
    ids64 = O.select(L64, K)
    tie = near_tie_mask(L64, K)
    assert np.array_equal(ids.cpu().numpy()[~tie], ids64[~tie])
    assert tie.sum() <= max(2, N // 50)


@pytest.mark.parametrize("N", [128, 16])
def test_route_tie_break_lowest_index(moe, N):
    # duplicate gate rows give bit-identical logits: the lower index must win
    # (tensor-core logits at 128 tokens, CUDA-core logits at 16)
    gen = torch.Generator().manual_seed(9)
    D, E, K = 128, 16, 4
    x = _bf16((N, D), gen)
    wg = _bf16((E, D), gen, D ** -0.5)
    wg[9] = wg[2]
    wg[15] = wg[2]
    wg[4] = wg[0]
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids, _ = moe.moe_route(x.cuda(), wg.cuda(), None, K, 0, logits_out=L)
    Lc = L.cpu()
    assert torch.equal(Lc[:, 2], Lc[:, 9]) and torch.equal(Lc[:, 2], Lc[:, 15])
    r = O.route_from_logits(Lc.numpy().astype(np.float64), K, 0)
    assert np.array_equal(ids.cpu().numpy(), r["ids"])
    for row in ids.cpu().tolist():
        for a, b in ((2, 9), (9, 15), (0, 4)):
            if a in row and b in row:
                assert row.index(a) < row.index(b)


# ------------------------------------------------------------------ grouped FFN
def _ffn_case(moe, counts, D, Dff, act, seed):
    gen = torch.Generator().manual_seed(seed)
    E = len(counts)
    rows = int(sum(counts))
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    xp = _bf16((rows, D), gen)
    w1 = _bf16((E, Dff, D), gen, D ** -0.5)
    w3 = _bf16((E, Dff, D), gen, D ** -0.5) if act == 1 else None
    w2 = _bf16((E, D, Dff), gen, Dff ** -0.5)
    ws = moe.workspace("ffn", rows, D, E, 1, Dff)
    h, y = moe.moe_grouped_ffn(xp.cuda(), off.cuda(), w1.cuda(), None if w3 is None else w3.cuda(),
                               w2.cuda(), act, ws=ws)
    _no_device_error(moe, ws)
    hg, yg = bits(h), bits(y)
    h_ref = np.zeros((rows, Dff))
    y_ref = np.zeros((rows, D))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        h_ref[a:b] = O.expert_up(bits(xp[a:b]), bits(w1[e]), None if w3 is None else bits(w3[e]), act)
        y_ref[a:b] = O.expert_down(hg[a:b], bits(w2[e]))     # GEMM2 on the GPU's own bf16 h
    assert_close(O.bf16_to_f64(hg), h_ref, "h")
    assert_close(O.bf16_to_f64(yg), y_ref, "y_perm")
    # h is one bf16 rounding of an fp32 value close to the fp64 one
    assert np.all(np.abs(O.bf16_to_f64(hg) - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 2e-3 * np.abs(h_ref).max())


# execution modes of the grouped FFN, forced through the library's tuning
# variables so every kernel variant meets the oracle
FFN_MODES = {
    "auto": {},
    "one": {"MOE_SWAP_GEMM": "0", "MOE_PAIR_GEMM": "0"},
    "one_n64": {"MOE_SWAP_GEMM": "0", "MOE_PAIR_GEMM": "0", "MOE_FFN_TILE_N": "64"},
    "one_n128": {"MOE_SWAP_GEMM": "0", "MOE_PAIR_GEMM": "0", "MOE_FFN_TILE_N": "128"},
    "one_n256": {"MOE_SWAP_GEMM": "0", "MOE_PAIR_GEMM": "0", "MOE_FFN_TILE_N": "256"},
    "swap": {"MOE_SWAP_GEMM": "1"},
}


@pytest.mark.parametrize("counts,D,Dff,act", [
    ([0, 1, 127, 129, 300], 128, 256, 1),
    ([0, 1, 127, 129, 300], 128, 256, 0),
    ([64], 128, 256, 0),
    ([5, 0, 0, 260, 3], 192, 192, 1),
    ([1, 2, 3, 4, 5, 6, 7, 8], 512, 768, 1),
    ([200, 0, 57, 384], 256, 128, 1),
    ([129] * 3, 64, 64, 0),
    ([3, 5], 1024, 512, 1),        # few tiles: split-K with fp32 partials
    ([3, 5], 1024, 512, 0),
])
@pytest.mark.parametrize("mode", list(FFN_MODES))
def test_grouped_ffn_matches_oracle(moe, counts, D, Dff, act, mode, monkeypatch):
    for k, v in FFN_MODES[mode].items():
        monkeypatch.setenv(k, v)
    _ffn_case(moe, counts, D, Dff, act, seed=len(counts) * 100 + D + Dff + act)


@pytest.mark.parametrize("counts,D,Dff,act", [
    ([300, 0, 513, 1, 256], 256, 256, 1),      # ragged 256-row pair tiles, both GEMMs paired
    ([700, 900, 3, 258], 512, 1024, 1),        # more pair tiles than resident clusters
    ([1, 2, 255, 257], 256, 128, 1),
    ([512, 0, 100], 512, 256, 0),              # SiLU: GEMM1 one-CTA, GEMM2 paired
])
def test_grouped_ffn_on_cta_pairs_matches_oracle(moe, counts, D, Dff, act, monkeypatch):
    monkeypatch.setenv("MOE_PAIR_GEMM", "1")
    _ffn_case(moe, counts, D, Dff, act, seed=7 * len(counts) + D + Dff + act)


# The mixed CTA-pair kernel (opt-in, MOE_PAIR_COLD_ROWS=n): experts with more
# than n rows on 256-row pair tiles, heaviest first; experts with fewer on
# weight-streaming tiles (weights as the MMA's M, 32 tokens as its N) spread
# among them in the same launch.
_MIXED16 = [0, 1, 31, 32, 33, 64, 65, 300, 513, 7, 0, 100, 2, 256, 257, 40]
_COLD16 = [3, 40, 64, 1, 17, 0, 9, 64, 2, 33, 50, 6, 1, 1, 60, 20]
_HOT16 = [300, 700, 65, 129, 256, 1024, 80, 99, 500, 70, 600, 66, 900, 400, 77, 200]
# 8 hot experts and 40 cold ones (0..64 rows) in shuffled order: about ten
# waves of tiles over the resident pairs
_MIXED48 = [int(c) for c in np.random.default_rng(48).permutation(
    [3000, 1500, 900, 600, 400, 300, 200, 150] + list(np.random.default_rng(49).integers(0, 65, 40)))]


@pytest.mark.parametrize("counts,D,Dff,act,cold", [
    (_MIXED16, 256, 256, 1, "64"),      # hot and cold experts in both GEMMs
    (_MIXED16, 512, 1024, 1, "64"),     # several cold stages per tile
    (_MIXED16, 256, 256, 0, "64"),      # SiLU: GEMM1 one-CTA, GEMM2 mixed
    (_COLD16, 512, 256, 1, "64"),       # cold experts only
    (_HOT16, 256, 512, 1, "64"),        # hot experts only (heaviest first)
    (_MIXED16, 256, 256, 1, "128"),     # up to four token tiles per cold expert
    (_MIXED16, 256, 256, 1, "1"),       # only one-row experts cold
    (_MIXED48, 512, 1024, 1, "64"),     # more tiles than resident clusters, skewed
])
def test_grouped_ffn_mixed_pairs_matches_oracle(moe, counts, D, Dff, act, cold, monkeypatch):
    monkeypatch.setenv("MOE_PAIR_GEMM", "1")
    monkeypatch.setenv("MOE_SWAP_GEMM", "0")
    monkeypatch.setenv("MOE_PAIR_COLD_ROWS", cold)
    _ffn_case(moe, counts, D, Dff, act, seed=11 * len(counts) + D + Dff + act)


# The pair kernels' tile list: experts heaviest first, each expert's m-tiles
# in bands (8 by default; MOE_PAIR_BAND pins the width).  Experts of several
# bands, a partial last band, and widths from 1 (n-tiles innermost) up.
_BANDS = [3000, 0, 2049, 1, 4100, 255, 257, 700]


@pytest.mark.parametrize("band", ["1", "3", "0", "64"])
def test_grouped_ffn_pair_bands_match_oracle(moe, band, monkeypatch):
    monkeypatch.setenv("MOE_PAIR_GEMM", "1")
    monkeypatch.setenv("MOE_SWAP_GEMM", "0")
    monkeypatch.setenv("MOE_PAIR_BAND", band)
    _ffn_case(moe, _BANDS, 256, 512, 1, seed=int(band) + 900)


def test_grouped_ffn_pairs_over_256_experts(moe, monkeypatch):
    # more experts than the heaviest-first sort and the mixed kernel handle:
    # the plain pair kernel, experts in index order
    monkeypatch.setenv("MOE_PAIR_GEMM", "1")
    monkeypatch.setenv("MOE_SWAP_GEMM", "0")
    monkeypatch.setenv("MOE_PAIR_COLD_ROWS", "64")
    counts = [int(c) for c in np.random.default_rng(300).integers(0, 160, 300)]
    _ffn_case(moe, counts, 256, 128, 1, seed=300)


def test_grouped_ffn_mixed_pairs_bitwise_equal_to_pair_tiles(moe, monkeypatch):
    """Weight-streaming tiles sum each output over K in the same order as the
    256-row pair tiles (16 products per MMA, k-blocks ascending), and the tile
    order never changes a sum: the mixed kernel and every band width give the
    bits of the plain pair kernel, cold experts included."""
    gen = torch.Generator().manual_seed(5)
    counts, D, Dff = _MIXED16, 512, 256
    E, rows = len(counts), sum(counts)
    off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32).cuda()
    xp = _bf16((rows, D), gen).cuda()
    w1 = _bf16((E, Dff, D), gen, D ** -0.5).cuda()
    w3 = _bf16((E, Dff, D), gen, D ** -0.5).cuda()
    w2 = _bf16((E, D, Dff), gen, Dff ** -0.5).cuda()
    monkeypatch.setenv("MOE_PAIR_GEMM", "1")
    monkeypatch.setenv("MOE_SWAP_GEMM", "0")
    res = {}
    # plain pair kernel in three band widths, then the mixed kernel
    for key, cold, band in (("plain", "0", "0"), ("band1", "0", "1"), ("band64", "0", "64"), ("mixed", "64", "0")):
        monkeypatch.setenv("MOE_PAIR_COLD_ROWS", cold)
        monkeypatch.setenv("MOE_PAIR_BAND", band)
        ws = moe.workspace("ffn", rows, D, E, 1, Dff)
        res[key] = moe.moe_grouped_ffn(xp, off, w1, w3, w2, 1, ws=ws)
        _no_device_error(moe, ws)
    for key in ("band1", "band64", "mixed"):
        assert torch.equal(res["plain"][0], res[key][0]) and torch.equal(res["plain"][1], res[key][1]), key


def test_grouped_ffn_rejects_bad_offsets(moe):
    D, Dff = 64, 64
    off = torch.tensor([0, 10, 5], dtype=torch.int32).cuda()            # decreasing
    xp = torch.zeros((10, D), dtype=torch.bfloat16).cuda()
    w = torch.zeros((2, Dff, D), dtype=torch.bfloat16).cuda()
    ws = moe.workspace("ffn", 10, D, 2, 1, Dff)
    moe.moe_grouped_ffn(xp, off, w, w, w, 1, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_ERR_DEVICE_BOUNDS


# ------------------------------------------------------------------ whole layer, small
@pytest.mark.parametrize("N,D,E,K,Dff,act,mode,zipf", [
    (64, 128, 8, 2, 256, 0, 0, 0.0),          # the tiny workload
    (1, 128, 8, 2, 256, 1, 0, 0.0),
    (77, 256, 16, 4, 192, 1, 1, 0.0),
    (300, 128, 32, 8, 128, 1, 1, 1.2),
    (130, 64, 1, 1, 64, 1, 0, 0.0),
    (50, 128, 4, 4, 128, 1, 1, 0.0),          # K = E: every token goes to every expert
    (20, 128, 64, 32, 128, 1, 0, 0.0),        # K at its maximum, 32
])
def test_layer_matches_oracle(moe, N, D, E, K, Dff, act, mode, zipf):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.Workload("t", N, D, E, K, Dff, act, mode, zipf)
    inp = synth.make_inputs(wl, seed=N + E)
    dev = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    ws = moe.workspace("layer", N, D, E, K, Dff)
    out = moe.moe_layer_forward(dev["x"], dev["w_gate"], dev["bias"], dev["w1"], dev["w3"], dev["w2"],
                                K, mode, act, ws=ws)
    _no_device_error(moe, ws)
    mid = moe.layer_intermediates(ws, N, D, E, K, Dff)
    # routing on the GPU's own logits (recomputed by moe_route; same kernel)
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids2, _ = moe.moe_route(dev["x"], dev["w_gate"], dev["bias"], K, mode, logits_out=L)
    assert torch.equal(ids2, mid["topk_ids"])
    r = O.route_from_logits(L.cpu().numpy().astype(np.float64), K, mode)
    assert np.array_equal(mid["topk_ids"].cpu().numpy(), r["ids"])
    assert np.max(np.abs(mid["topk_w"].cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    assert np.array_equal(mid["expert_offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(mid["perm_src"].cpu().numpy(), r["perm_src"])
    assert np.array_equal(mid["inv_perm"].cpu().numpy(), r["inv_perm"])
    # FFN + combine in fp64 on the GPU's routing
    xb = bits(inp["x"])
    y = O.grouped_ffn(O.gather_rows(xb, r["perm_src"]), r["offsets"], bits(inp["w1"]),
                      None if inp["w3"] is None else bits(inp["w3"]), bits(inp["w2"]), act)
    ref = O.combine(y, r["inv_perm"], r["w"])
    assert_close(f64(out), ref, "out")
    # and the whole chain of the oracle, from its own fp64 logits
    b64 = None if inp["bias"] is None else inp["bias"].numpy().astype(np.float64)
    full = O.layer(xb, bits(inp["w_gate"]), b64, bits(inp["w1"]),
                   None if inp["w3"] is None else bits(inp["w3"]), bits(inp["w2"]), K, mode, act)
    tie = near_tie_mask(full["logits"], K)
    assert_close(f64(out)[~tie], full["out"][~tie], "out vs full oracle")


# ------------------------------------------------------------------ routing statistics
@pytest.mark.parametrize("E,step", [(8, 0.1), (256, -0.05), (1000, 0.1)])
def test_routing_stats_matches_oracle(moe, E, step):
    gen = torch.Generator().manual_seed(E)
    ema = torch.softmax(torch.randn(E, generator=gen), 0).to(torch.float32)
    bias = torch.randn(E, generator=gen).to(torch.float32)
    ema_d, bias_d = ema.cuda(), bias.cuda()
    ema_o, bias_o = ema.numpy().astype(np.float64), bias.numpy().astype(np.float64)
    for it in range(3):   # three batches in a row
        counts = torch.randint(0, 50, (E,), generator=gen)
        off = torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(counts, 0)]).to(torch.int32)
        kl = moe.moe_routing_stats(off.cuda(), ema_d, bias_d, decay=0.99, bias_step=step)
        ema_o, bias_o, kl_o = O.routing_stats(off.numpy(), ema_o, bias_o, 0.99, step)
        np.testing.assert_allclose(ema_d.cpu().numpy(), ema_o, rtol=1e-5, atol=1e-8)
        np.testing.assert_allclose(bias_d.cpu().numpy(), bias_o, rtol=1e-5, atol=1e-6)
        assert abs(kl.item() - kl_o) <= 1e-5 * max(1.0, abs(kl_o))
    # a batch without assignments changes nothing
    before = ema_d.clone()
    moe.moe_routing_stats(torch.zeros(E + 1, dtype=torch.int32, device="cuda"), ema_d, bias_d)
    assert torch.equal(before, ema_d)


# ------------------------------------------------------------------ route + permute in one call
@pytest.mark.parametrize("N,D,E,K,mode,with_bias", [
    (1, 2048, 128, 8, 0, False),      # one decode token: top-K and permutation in one launch
    (8, 2048, 128, 8, 1, True),       # up to 8 tokens fused
    (8, 128, 32, 32, 0, False),       # 256 assignments, the largest fused call
    (3, 128, 8, 2, 0, False),
    (6, 128, 1024, 12, 1, True),      # 1024 experts fused
    (32, 256, 128, 8, 0, True),       # more tokens: the separate launches
    (128, 256, 16, 2, 1, False),      # logits from the tensor-core GEMM (N > 32)
])
def test_route_permute_equals_route_then_permute(moe, N, D, E, K, mode, with_bias):
    gen = torch.Generator().manual_seed(N * 7 + E + K)
    x = _bf16((N, D), gen).cuda()
    wg = _bf16((E, D), gen, D ** -0.5).cuda()
    bias = (torch.randn(E, generator=gen) * 0.5).float().cuda() if with_bias else None
    got = moe.moe_route_permute(x, wg, bias, K, mode)
    ids, w = moe.moe_route(x, wg, bias, K, mode)
    ref = (ids, w) + moe.moe_permute(x, ids, E)
    torch.cuda.synchronize()
    for name, a, b in zip(("topk_ids", "topk_w", "expert_offsets", "perm_src", "inv_perm", "x_perm"), got, ref):
        assert torch.equal(a, b), name
    # and the oracle's selection and placement on the GPU's own fp32 logits
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    moe.moe_route(x, wg, bias, K, mode, logits_out=L)
    r = O.route_from_logits(L.cpu().numpy().astype(np.float64), K, mode)
    assert np.array_equal(got[0].cpu().numpy(), r["ids"])
    assert np.max(np.abs(got[1].cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    for key, i in (("offsets", 2), ("perm_src", 3), ("inv_perm", 4)):
        assert np.array_equal(got[i].cpu().numpy(), r[key]), key
    assert np.array_equal(bits(got[5]), O.gather_rows(bits(x), r["perm_src"]))


def test_route_permute_zero_tokens(moe):
    E, D, K = 16, 128, 2
    x = torch.zeros((0, D), dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros((E, D), dtype=torch.bfloat16, device="cuda")
    off = torch.full((E + 1,), 7, dtype=torch.int32, device="cuda")
    got = moe.moe_route_permute(x, wg, None, K, 0, expert_offsets=off)
    torch.cuda.synchronize()
    assert torch.all(got[2] == 0)


@pytest.mark.parametrize("N,E,K", [(1, 128, 8), (8, 128, 8), (5, 64, 4)])
def test_layer_with_fused_route_permute_equals_separate_launches(moe, N, E, K, monkeypatch):
    from mixture_experts_layer_02_gb300 import synth
    monkeypatch.setenv("MOE_LAYER_DECODE", "0")   # the chain of launches, with and without the fusion
    wl = synth.Workload("d", N, 256, E, K, 128, 1, 0, 0.0)
    inp = {k: (None if v is None else v.cuda()) for k, v in synth.make_inputs(wl, seed=N).items()}
    outs = []
    for flag in ("1", "0"):
        monkeypatch.setenv("MOE_FUSED_ROUTE_PERMUTE", flag)
        ws = moe.workspace("layer", N, 256, E, K, 128)
        outs.append(moe.moe_layer_forward(inp["x"], inp["w_gate"], None, inp["w1"], inp["w3"], inp["w2"],
                                          K, 0, 1, ws=ws))
        _no_device_error(moe, ws)
    assert torch.equal(outs[0], outs[1])


# ------------------------------------------------------------------ launch accounting
@pytest.mark.parametrize("N,D,E,K,Dff,cap", [(64, 128, 8, 2, 256, -1), (4, 2048, 128, 8, 768, -1),
                                             (8, 256, 16, 8, 128, -1), (1, 2048, 128, 8, 768, -1),
                                             (700, 256, 16, 8, 128, -1), (300, 128, 32, 8, 128, 40)])
def test_layer_launch_count_is_what_runs(moe, N, D, E, K, Dff, cap, tmp_path):
    # capture one layer call in a CUDA graph and count its kernel nodes
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.Workload("c", N, D, E, K, Dff, 1, 0, 0.0)
    inp = {k: (None if v is None else v.cuda()) for k, v in synth.make_inputs(wl, seed=1).items()}
    if cap < 0:
        ws = moe.workspace("layer", N, D, E, K, Dff)
        run = lambda: moe.moe_layer_forward(inp["x"], inp["w_gate"], None, inp["w1"], inp["w3"], inp["w2"],
                                            K, 0, 1, ws=ws)
    else:
        ws = moe.workspace_padded("layer", N, D, E, K, Dff, cap)
        run = lambda: moe.moe_layer_forward_padded(inp["x"], inp["w_gate"], None, inp["w1"], inp["w3"],
                                                   inp["w2"], K, 0, 1, cap, ws=ws)
    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph(keep_graph=True)
    with torch.cuda.graph(g):
        run()
    assert _graph_kernel_nodes(g.raw_cuda_graph()) == moe.layer_launches(N, D, E, K, Dff, 1, cap)


def _graph_kernel_nodes(graph_handle: int) -> int:
    """Kernel nodes of a captured graph, counted through the driver API."""
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(ctypes.c_void_p(graph_handle), None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * n.value)()
    assert cu.cuGraphGetNodes(ctypes.c_void_p(graph_handle), nodes, ctypes.byref(n)) == 0
    kinds = []
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kinds.append(t.value)
    return sum(1 for t in kinds if t == 0)   # CU_GRAPH_NODE_TYPE_KERNEL
