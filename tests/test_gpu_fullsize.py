"""Full-size parity: every workload at its real size, through moe_layer_forward
(the call the benchmark's end-to-end leg times, same launch configuration).

Routing and permutation are checked on ALL tokens (ids, weights, offsets,
perm_src, inv_perm against the oracle run on the GPU's own fp32 logits).
The FFN and the output are checked on sampled rows and tokens that the oracle
computes one by one, with the expert weights those rows use copied to the
host.  The decode workloads (N <= 256) are checked on every token.
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

    experts = HostExperts(inp)
    rows = r["inv_perm"][toks].ravel()
    xp = bits(mid["x_perm"][torch.as_tensor(rows, device="cuda", dtype=torch.long)])
    assert np.array_equal(xp, np.repeat(xb, K, axis=0))          # x_perm rows are bit copies
    h_gpu = bits(mid["h"][torch.as_tensor(rows, device="cuda", dtype=torch.long)])
    y_gpu = bits(mid["y_perm"][torch.as_tensor(rows, device="cuda", dtype=torch.long)])
    h_ref = np.empty((len(rows), Dff))
    y_ref = np.empty((len(rows), D))          # GEMM2 from the GPU's bf16 h
    y64 = np.empty((len(rows), D))            # fp64 chain from x
    for i, (t, k) in enumerate([(t, k) for t in range(len(toks)) for k in range(K)]):
        e = int(r["ids"][toks[t], k])
        w1e, w3e, w2e = experts(e)
        h_ref[i] = O.expert_up(xb[t:t + 1], w1e, w3e, wl.act)[0]
        y_ref[i] = O.expert_down(h_gpu[i:i + 1], w2e)[0]
        y64[i] = O.expert_down(h_ref[i:i + 1], w2e)[0]
    assert_close(O.bf16_to_f64(h_gpu), h_ref, f"{name} h")
    assert_close(O.bf16_to_f64(y_gpu), y_ref, f"{name} y_perm")
    local_rows = np.arange(len(rows), dtype=np.int32).reshape(len(toks), K)
    ref = O.combine(y64, local_rows, r["w"][toks])
    m = assert_close(f64(out[torch.as_tensor(toks, device="cuda")]), ref, f"{name} out")
    print(f"{name}: tokens checked={len(toks)} near_ties={int(tie.sum())} "
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
