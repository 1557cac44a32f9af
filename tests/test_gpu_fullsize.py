"""Full-size parity: every workload at its real size, through moe_layer_forward
(the call the benchmark's end-to-end leg times, same launch configuration).

Routing and permutation are checked on ALL tokens (ids, weights, offsets,
perm_src, inv_perm against the oracle run on the GPU's own fp32 logits).

The grouped FFN is checked on stratified permuted rows, complete rows of h
and y_perm: every expert's first and last row and two rows (one in each
64-row half) of every 128-row block of every expert's segment.  Tiles start
at segment starts, so this touches every m-tile of the 256-row CTA-pair
tiling and of the 128-row one-CTA tiling, every epilogue lane half, every
wave of the persistent schedule and both TMEM accumulators.  h is compared
with the oracle's expert FFN applied to the same x_perm row, y_perm with the
oracle's GEMM2 applied to the GPU's own bf16 h (so a failure points at one
GEMM).  The decode workloads (N <= 256) are checked on every row.  The layer
output is checked on sampled tokens (all of them for decode) against the
oracle's fp64 chain.
"""
import numpy as np
import pytest
import torch

from helpers import WEIGHT_ATOL, assert_close, bits, f64, logits_bound, near_tie_mask
from oracle import oracle as O

pytestmark = pytest.mark.gpu

SAMPLE = {"mixtral": 16, "dsv3": 6, "dsv3_zipf": 6}


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


class HostExperts:
    """Host copies of single experts' weights, fetched on demand."""

    def __init__(self, inp):
        self.inp = inp
        self.cache = {}

    def __call__(self, e):
        if e not in self.cache:
            w3 = self.inp["w3"]
            self.cache[e] = (bits(self.inp["w1"][e]), None if w3 is None else bits(w3[e]),
                             bits(self.inp["w2"][e]))
        return self.cache[e]


def stratified_rows(off, rng, block=128):
    """Permuted rows to check: each expert's first and last row and, in every
    `block`-row block of its segment (blocks start at the segment start, as
    the kernels' m-tiles do), one random row in each half of the block."""
    rows = set()
    for e in range(len(off) - 1):
        a, b = int(off[e]), int(off[e + 1])
        if a == b:
            continue
        rows.update((a, b - 1))
        for t0 in range(a, b, block):
            for h0 in (t0, t0 + block // 2):
                h1 = min(h0 + block // 2, b)
                if h0 < h1:
                    rows.add(int(rng.integers(h0, h1)))
    return np.array(sorted(rows), np.int64)


def tiles_covered(off, rows, tile):
    """(tiles holding a checked row, all tiles) of a `tile`-row m-tiling."""
    seg = np.searchsorted(off, rows, side="right") - 1
    hit = set(zip(seg.tolist(), ((rows - off[seg]) // tile).tolist()))
    total = sum(-(-int(off[e + 1] - off[e]) // tile) for e in range(len(off) - 1))
    return len(hit), total


def _run(moe, name):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.WORKLOADS[name]
    torch.cuda.empty_cache()
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    N, D, E, K, Dff = wl.N, wl.D, wl.E, wl.K, wl.Dff
    ws = moe.workspace("layer", N, D, E, K, Dff)
    out = moe.moe_layer_forward(inp["x"], inp["w_gate"], inp["bias"], inp["w1"], inp["w3"], inp["w2"],
                                K, wl.mode, wl.act, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    return wl, inp, ws, out


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "dsv3_zipf", "qwen3_N1", "qwen3_N8",
                                  "qwen3_N32", "qwen3_N128", "qwen3_N256"])
def test_fullsize_layer(moe, name):
    wl, inp, ws, out = _run(moe, name)
    N, D, E, K, Dff = wl.N, wl.D, wl.E, wl.K, wl.Dff
    mid = moe.layer_intermediates(ws, N, D, E, K, Dff)

    # ---- routing + permutation, every token, on the GPU's own fp32 logits
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids2, w2g = moe.moe_route(inp["x"], inp["w_gate"], inp["bias"], K, wl.mode, logits_out=L)
    assert torch.equal(ids2, mid["topk_ids"]) and torch.equal(w2g, mid["topk_w"])
    Lg = L.cpu().numpy().astype(np.float64)
    r = O.route_from_logits(Lg, K, wl.mode)
    assert np.array_equal(mid["topk_ids"].cpu().numpy(), r["ids"])
    assert np.max(np.abs(mid["topk_w"].cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    assert np.array_equal(mid["expert_offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(mid["perm_src"].cpu().numpy(), r["perm_src"])
    assert np.array_equal(mid["inv_perm"].cpu().numpy(), r["inv_perm"])

    # ---- sampled tokens (all of them for decode)
    rng = np.random.default_rng(N)
    if N <= 256:
        toks = np.arange(N)
    else:
        toks = np.unique(np.concatenate([[0, N - 1], rng.choice(N, SAMPLE[name] - 2, replace=False)]))
    xb = bits(inp["x"][torch.as_tensor(toks, device="cuda")])
    b64 = None if inp["bias"] is None else inp["bias"].cpu().numpy().astype(np.float64)
    # end-to-end routing from the oracle's fp64 logits, near-ties reported apart
    L64 = O.logits(xb, bits(inp["w_gate"]), b64)
    tie = near_tie_mask(L64, K)
    assert np.array_equal(O.select(L64, K)[~tie], r["ids"][toks][~tie])
    assert np.all(np.abs(Lg[toks] - L64) <= logits_bound(O.bf16_to_f64(xb), f64(inp["w_gate"]), b64))

    # ---- grouped FFN on stratified permuted rows (every row for decode),
    # complete rows of h and y_perm, expert by expert
    off = r["offsets"]
    prow = np.arange(N * K) if N <= 256 else stratified_rows(off, rng)
    sel = torch.as_tensor(prow, device="cuda", dtype=torch.long)
    xp = bits(mid["x_perm"][sel])
    assert np.array_equal(xp, bits(inp["x"][torch.as_tensor(r["perm_src"][prow], device="cuda",
                                                            dtype=torch.long)]))   # bit copies of x rows
    h_gpu = bits(mid["h"][sel])
    y_gpu = bits(mid["y_perm"][sel])
    h_ref = np.empty((len(prow), Dff))
    y_ref = np.empty((len(prow), D))          # GEMM2 from the GPU's bf16 h
    seg = np.searchsorted(off, prow, side="right") - 1
    for e in np.unique(seg):
        i = np.nonzero(seg == e)[0]
        w3 = inp["w3"]
        w1e, w3e, w2e = bits(inp["w1"][e]), None if w3 is None else bits(w3[e]), bits(inp["w2"][e])
        h_ref[i] = O.expert_up(xp[i], w1e, w3e, wl.act)
        y_ref[i] = O.expert_down(h_gpu[i], w2e)
    mh = assert_close(O.bf16_to_f64(h_gpu), h_ref, f"{name} h")
    my = assert_close(O.bf16_to_f64(y_gpu), y_ref, f"{name} y_perm")
    cov128, all128 = tiles_covered(off, prow, 128)
    cov256, all256 = tiles_covered(off, prow, 256)
    assert cov128 == all128 and cov256 == all256

    # ---- the layer output on sampled tokens, fp64 chain from x
    experts = HostExperts(inp)
    y64 = np.empty((len(toks) * K, D))
    for i, (t, k) in enumerate([(t, k) for t in range(len(toks)) for k in range(K)]):
        w1e, w3e, w2e = experts(int(r["ids"][toks[t], k]))
        y64[i] = O.expert_down(O.expert_up(xb[t:t + 1], w1e, w3e, wl.act), w2e)[0]
    local_rows = np.arange(len(toks) * K, dtype=np.int32).reshape(len(toks), K)
    ref = O.combine(y64, local_rows, r["w"][toks])
    m = assert_close(f64(out[torch.as_tensor(toks, device="cuda")]), ref, f"{name} out")
    print(f"{name}: permuted rows checked={len(prow)} of {N * K} (128-row tiles {cov128}/{all128}, "
          f"256-row tiles {cov256}/{all256}) h rel_frob={mh['rel_frob']:.3e} y rel_frob={my['rel_frob']:.3e}; "
          f"tokens checked={len(toks)} near_ties={int(tie.sum())} "
          f"max_abs={m['max_abs']:.3e} max_ref={m['max_ref']:.3e} rel_frob={m['rel_frob']:.3e}")


@pytest.mark.parametrize("name", ["mixtral", "dsv3"])
def test_fullsize_fused_equals_unfused(moe, name, monkeypatch):
    """At full size the layer with the permutation fused into GEMM1
    (MOE_GATHER=1) gives the same bits as the row copy + unfused GEMM1."""
    wl, inp, ws, out = _run(moe, name)
    monkeypatch.setenv("MOE_GATHER", "1")
    out0 = moe.moe_layer_forward(inp["x"], inp["w_gate"], inp["bias"], inp["w1"], inp["w3"], inp["w2"],
                                 wl.K, wl.mode, wl.act, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    assert torch.equal(out, out0)


@pytest.mark.parametrize("name", ["mixtral", "dsv3_zipf"])
def test_fullsize_deterministic(moe, name):
    wl, inp, ws, out = _run(moe, name)
    out2 = moe.moe_layer_forward(inp["x"], inp["w_gate"], inp["bias"], inp["w1"], inp["w3"], inp["w2"],
                                 wl.K, wl.mode, wl.act, ws=ws)
    assert torch.equal(out, out2)
