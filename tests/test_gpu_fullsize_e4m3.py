"""Full-size parity of the FP8 (e4m3) layer: every workload at its real size,
through moe_layer_forward_e4m3 (the call the benchmark's end-to-end leg times).

Routing, permutation and the token codes are checked on ALL tokens.  The FFN
and the output are checked on sampled tokens, one by one, with the oracle's
own e4m3 codes of the experts those tokens use (equal, bit for bit, to the
GPU's codes of the same experts).  Decode workloads (N <= 256) are checked on
every token."""
import numpy as np
import pytest
import torch

from helpers import WEIGHT_ATOL, assert_close, bits, f64
from oracle import oracle as O

pytestmark = pytest.mark.gpu

SAMPLE = {"mixtral": 12, "dsv3": 6, "dsv3_zipf": 6}


@pytest.fixture(scope="module")
def moe(cuda_device):
    from mixture_experts_layer_02_gb300 import build, moe as m
    build.build()
    m.load()
    return m


def _u8(t):
    return t.detach().contiguous().cpu().numpy()


class OracleExperts:
    """The oracle's e4m3 codes and scales of single experts, checked against
    the GPU's codes of the same expert when first fetched."""

    def __init__(self, inp, qw):
        self.inp, self.qw, self.cache = inp, qw, {}

    def __call__(self, e):
        if e not in self.cache:
            w1q, s1 = O.quant_rows_e4m3(bits(self.inp["w1"][e]))
            w2q, s2 = O.quant_rows_e4m3(bits(self.inp["w2"][e]))
            assert np.array_equal(w1q, _u8(self.qw["w1q"][e])) and np.array_equal(s1, _u8(self.qw["s1"][e]))
            assert np.array_equal(w2q, _u8(self.qw["w2q"][e])) and np.array_equal(s2, _u8(self.qw["s2"][e]))
            w3q = s3 = None
            if self.inp["w3"] is not None:
                w3q, s3 = O.quant_rows_e4m3(bits(self.inp["w3"][e]))
                assert np.array_equal(w3q, _u8(self.qw["w3q"][e])) and np.array_equal(s3, _u8(self.qw["s3"][e]))
            self.cache[e] = (w1q, s1, w3q, s3, w2q, s2)
        return self.cache[e]


@pytest.mark.parametrize("name", ["mixtral", "dsv3", "dsv3_zipf", "qwen3_N1", "qwen3_N8",
                                  "qwen3_N32", "qwen3_N128", "qwen3_N256"])
def test_fullsize_layer_e4m3(moe, name):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.WORKLOADS[name]
    N, D, E, K, Dff = wl.N, wl.D, wl.E, wl.K, wl.Dff
    torch.cuda.empty_cache()
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
    ws = moe.workspace("layer_e4m3", N, D, E, K, Dff)
    out = moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], inp["bias"], qw, K, wl.mode, wl.act, ws=ws)
    assert moe.read_device_error(ws) == moe.MOE_OK
    mid = moe.layer_e4m3_intermediates(ws, N, D, E, K, Dff)

    # ---- routing + permutation, every token, on the GPU's own fp32 logits
    L = torch.empty((N, E), dtype=torch.float32, device="cuda")
    ids2, _ = moe.moe_route(inp["x"], inp["w_gate"], inp["bias"], K, wl.mode, logits_out=L)
    assert torch.equal(ids2, mid["topk_ids"])
    r = O.route_from_logits(L.cpu().numpy().astype(np.float64), K, wl.mode)
    assert np.array_equal(mid["topk_ids"].cpu().numpy(), r["ids"])
    assert np.max(np.abs(mid["topk_w"].cpu().numpy() - r["w"])) <= WEIGHT_ATOL
    assert np.array_equal(mid["expert_offsets"].cpu().numpy(), r["offsets"])
    assert np.array_equal(mid["perm_src"].cpu().numpy(), r["perm_src"])
    assert np.array_equal(mid["inv_perm"].cpu().numpy(), r["inv_perm"])

    # ---- token codes, every token; permuted codes on the sampled rows
    xb_all = bits(inp["x"])
    o_xq, o_sx = O.quant_rows_e4m3(xb_all)
    assert np.array_equal(_u8(mid["xq"]), o_xq) and np.array_equal(_u8(mid["x_scale"]), o_sx)

    rng = np.random.default_rng(N + 1)
    toks = np.arange(N) if N <= 256 else \
        np.unique(np.concatenate([[0, N - 1], rng.choice(N, SAMPLE[name] - 2, replace=False)]))
    rows = r["inv_perm"][toks].ravel()
    trow = torch.as_tensor(rows, device="cuda", dtype=torch.long)
    assert np.array_equal(_u8(mid["xq_perm"][trow]), np.repeat(o_xq[toks], K, axis=0))
    h_gpu = bits(mid["h"][trow])
    hq_gpu, hs_gpu = _u8(mid["hq"][trow]), _u8(mid["h_scale"][trow])
    y_gpu = f64(mid["y_perm"][trow])

    experts = OracleExperts(inp, qw)
    h_ref = np.empty((len(rows), Dff))
    y_ref = np.empty((len(rows), D))          # GEMM2 on the GPU's codes of h
    y64 = np.empty((len(rows), D))            # the oracle's own FP8 chain
    for i, (t, k) in enumerate([(t, k) for t in range(len(toks)) for k in range(K)]):
        e = int(r["ids"][toks[t], k])
        w1q, s1, w3q, s3, w2q, s2 = experts(e)
        xq1, sx1 = o_xq[toks[t]:toks[t] + 1], o_sx[toks[t]:toks[t] + 1]
        g = O.grouped_ffn_e4m3(xq1, sx1, np.array([0, 1], np.int32), w1q[None], s1[None],
                               None if w3q is None else w3q[None], None if s3 is None else s3[None],
                               w2q[None], s2[None], wl.act)
        h_ref[i] = g["h"][0]
        y64[i] = g["y"][0]
        y_ref[i] = O.expert_down_e4m3(hq_gpu[i:i + 1], hs_gpu[i:i + 1], w2q, s2)[0]
    assert_close(O.bf16_to_f64(h_gpu), h_ref, f"{name} h")
    r_hq, r_hs = O.quant_rows_e4m3(h_gpu)
    assert np.array_equal(hq_gpu, r_hq) and np.array_equal(hs_gpu, r_hs)
    assert_close(y_gpu, y_ref, f"{name} y_perm")
    local_rows = np.arange(len(rows), dtype=np.int32).reshape(len(toks), K)
    ref = O.combine(y64, local_rows, r["w"][toks])
    m = assert_close(f64(out[torch.as_tensor(toks, device="cuda")]), ref, f"{name} out")
    print(f"{name} e4m3: tokens checked={len(toks)} max_abs={m['max_abs']:.3e} "
          f"max_ref={m['max_ref']:.3e} rel_frob={m['rel_frob']:.3e}")


def test_fullsize_e4m3_deterministic(moe):
    from mixture_experts_layer_02_gb300 import synth
    wl = synth.WORKLOADS["dsv3_zipf"]
    torch.cuda.empty_cache()
    inp = synth.make_inputs(wl, seed=0, device="cuda")
    qw = moe.quantize_experts_e4m3(inp["w1"], inp["w3"], inp["w2"])
    ws = moe.workspace("layer_e4m3", wl.N, wl.D, wl.E, wl.K, wl.Dff)
    a = moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], inp["bias"], qw, wl.K, wl.mode, wl.act, ws=ws)
    b = moe.moe_layer_forward_e4m3(inp["x"], inp["w_gate"], inp["bias"], qw, wl.K, wl.mode, wl.act, ws=ws)
    assert torch.equal(a, b)
