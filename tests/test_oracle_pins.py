"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Every check here uses an independent route to the answer: the pages' worked
example, closed forms, brute-force enumeration, numpy/torch library routines
on cases where they are exact or tie-free, and invariants of the mathematics.
Source for the method: "MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切"
(zoe.im), 第一层 (Router and Top-K) and 第二层 范式 A Steps 1-3.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a) -> np.ndarray:
    """Round an array to bf16 (RNE via torch) and return the raw bits."""
    t = torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(bits) -> np.ndarray:
    return O.bf16_to_f64(bits)


# ---------------------------------------------------------------- O4 / O5
def test_page_permutation_example():
    g = json.load(open(os.path.join(GOLDEN, "permutation_example.json")))
    E, K = g["num_experts"], g["top_k"]
    ids = np.array(g["assignment"], np.int32).reshape(-1, K)
    off = O.offsets(ids, E)
    assert off.tolist() == g["expert_offsets"]
    perm_src, inv_perm = O.place(ids, off, E)
    expected_perm = [t for seg in g["segments"] for t in seg]
    assert perm_src.tolist() == expected_perm
    for e, seg in enumerate(g["segments"]):
        assert perm_src[off[e]:off[e + 1]].tolist() == seg
    # inv_perm sends token t to the row that holds it
    for t in range(ids.shape[0]):
        assert perm_src[inv_perm[t, 0]] == t


@pytest.mark.parametrize("N,E,K,seed", [(1, 1, 1, 0), (37, 5, 3, 1), (200, 16, 4, 2), (0, 4, 2, 3)])
def test_offsets_are_prefix_sum_and_placement_inverts(N, E, K, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(N)]).astype(np.int32) if N else \
        np.zeros((0, K), np.int32)
    off = O.offsets(ids, E)
    counts = np.bincount(ids.ravel(), minlength=E)
    assert off[0] == 0 and off[-1] == N * K
    assert np.array_equal(np.diff(off), counts)
    perm_src, inv_perm = O.place(ids, off, E)
    # permute then un-permute is the identity on (t, k)
    for t in range(N):
        for k in range(K):
            r = inv_perm[t, k]
            assert perm_src[r] == t
            assert off[ids[t, k]] <= r < off[ids[t, k] + 1]
    # each segment lists its tokens in ascending order (stable)
    for e in range(E):
        seg = perm_src[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)
    # a row of x travels to every row that names it
    x = bf16(rng.standard_normal((N, 8)))
    xp = O.gather_rows(x, perm_src)
    for t in range(N):
        for k in range(K):
            assert np.array_equal(xp[inv_perm[t, k]], x[t])


def test_bad_ids_rejected():
    with pytest.raises(ValueError):
        O.offsets(np.array([[0], [3]], np.int32), 3)
    with pytest.raises(ValueError):
        O.select(np.zeros((2, 3)), 4)


# ---------------------------------------------------------------- O2
def _brute_topk(row, K):
    """The unique K-subset whose members all beat all non-members under the
    order (value desc, index asc), listed in that order -- by enumeration."""
    E = len(row)
    beats = lambda a, b: (row[a] > row[b]) or (row[a] == row[b] and a < b)
    found = []
    for S in itertools.combinations(range(E), K):
        rest = [e for e in range(E) if e not in S]
        if all(beats(a, b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1
    S = list(found[0])
    # order inside the subset: repeatedly the member that beats all others left
    ordered = []
    while S:
        top = [a for a in S if all(a == b or beats(a, b) for b in S)][0]
        ordered.append(top)
        S.remove(top)
    return ordered


@pytest.mark.parametrize("E,K", [(1, 1), (3, 1), (4, 2), (6, 3), (8, 2), (10, 3)])
def test_select_matches_brute_force_with_ties(E, K):
    rng = np.random.default_rng(E * 10 + K)
    # small integer logits: ties everywhere
    L = rng.integers(-2, 3, size=(300, E)).astype(np.float64)
    ids = O.select(L, K)
    for t in range(L.shape[0]):
        assert ids[t].tolist() == _brute_topk(L[t], K)


def test_select_tie_break_duplicate_gate_rows_and_signed_zero():
    rng = np.random.default_rng(7)
    D, E = 64, 6
    x = bf16(rng.standard_normal((5, D)))
    wg = bf16(rng.standard_normal((E, D)) / 8)
    wg[4] = wg[1]            # experts 1 and 4 have identical gates
    wg[5] = wg[0]            # experts 0 and 5 too
    L = O.logits(x, wg)
    assert np.array_equal(L[:, 1], L[:, 4]) and np.array_equal(L[:, 0], L[:, 5])
    ids = O.select(L, E)
    for t in range(5):
        r = ids[t].tolist()
        assert r.index(1) + 1 == r.index(4)       # equal logits: lower index first, adjacent
        assert r.index(0) + 1 == r.index(5)
    # -0.0 and +0.0 are equal: the index decides
    Z = np.array([[-0.0, 0.0, -1.0], [0.0, -0.0, -1.0]])
    assert O.select(Z, 2).tolist() == [[0, 1], [0, 1]]


def test_select_matches_torch_topk_on_tie_free_rows():
    rng = np.random.default_rng(3)
    L = rng.standard_normal((500, 256))
    for K in (1, 2, 8):
        ids = O.select(L, K)
        tv, ti = torch.topk(torch.from_numpy(L), K, dim=-1, sorted=True)
        assert np.array_equal(ids, ti.numpy().astype(np.int32))


# ---------------------------------------------------------------- O3
def test_weights_softmax_and_sigmoid_against_torch():
    rng = np.random.default_rng(11)
    L = rng.standard_normal((400, 32)) * 3
    for K in (1, 2, 8):
        ids = O.select(L, K)
        sel = torch.from_numpy(np.take_along_axis(L, ids.astype(np.int64), 1))
        w = O.weights(L, ids, O.SOFTMAX_TOPK)
        np.testing.assert_allclose(w, torch.softmax(sel, -1).numpy(), rtol=0, atol=1e-15)
        s = torch.sigmoid(sel)
        ws = O.weights(L, ids, O.SIGMOID_NORM)
        np.testing.assert_allclose(ws, (s / s.sum(-1, keepdim=True)).numpy(), rtol=0, atol=1e-15)
        for ww in (w, ws):
            assert np.max(np.abs(ww.sum(1) - 1.0)) <= 1e-15 * K
            if K == 1:
                assert np.all(ww == 1.0)


def test_weights_closed_forms():
    # two selected logits a, b: softmax weight of the first is 1/(1+e^(b-a))
    L = np.array([[2.0, 0.5, -1.0]])
    ids = O.select(L, 2)
    assert ids.tolist() == [[0, 1]]
    w = O.weights(L, ids, O.SOFTMAX_TOPK)
    assert w[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-1.5)), abs=1e-16)
    ws = O.weights(L, ids, O.SIGMOID_NORM)
    s0, s1 = 1 / (1 + math.exp(-2.0)), 1 / (1 + math.exp(-0.5))
    assert ws[0, 0] == pytest.approx(s0 / (s0 + s1), abs=1e-16)
    # every sigmoid underflows to 0: uniform weights
    Lu = np.full((1, 4), -1e6)
    wu = O.weights(Lu, O.select(Lu, 3), O.SIGMOID_NORM)
    assert np.allclose(wu, 1 / 3, atol=0)


# ---------------------------------------------------------------- O1
def test_logits_match_numpy_and_bias_shifts_exactly():
    rng = np.random.default_rng(5)
    N, D, E = 9, 96, 7
    x = bf16(rng.standard_normal((N, D)))
    wg = bf16(rng.standard_normal((E, D)) / math.sqrt(D))
    L = O.logits(x, wg)
    ref = f64(x) @ f64(wg).T
    np.testing.assert_allclose(L, ref, rtol=1e-13, atol=1e-13)
    bias = rng.standard_normal(E)
    Lb = O.logits(x, wg, bias)
    assert np.array_equal(Lb, L + bias[None, :])
    # a transposed or misindexed operand would break this exact small case
    x1 = np.zeros((1, D), np.float32); x1[0, 3] = 1.0
    wg1 = np.zeros((E, D), np.float32); wg1[:, 3] = np.arange(E)
    assert O.logits(bf16(x1), bf16(wg1)).tolist() == [list(map(float, range(E)))]


# ---------------------------------------------------------------- O6
def _dense_ffn(x, w1, w3, w2, act):
    g = f64(x) @ f64(w1).T
    h = g / (1 + np.exp(-g))
    if act == O.ACT_SWIGLU:
        h = h * (f64(x) @ f64(w3).T)
    return h, h @ f64(w2).T


@pytest.mark.parametrize("act", [O.ACT_SILU, O.ACT_SWIGLU])
def test_expert_ffn_single_expert_is_dense_ffn(act):
    rng = np.random.default_rng(17)
    N, D, Dff = 6, 64, 96                       # D != Dff catches a transposed W2
    x = bf16(rng.standard_normal((N, D)))
    w1 = bf16(rng.standard_normal((1, Dff, D)) / 8)
    w3 = bf16(rng.standard_normal((1, Dff, D)) / 8)
    w2 = bf16(rng.standard_normal((1, D, Dff)) / 10)
    h_ref, y_ref = _dense_ffn(x, w1[0], w3[0], w2[0], act)
    h = O.expert_up(x, w1[0], w3[0], act)
    np.testing.assert_allclose(h, h_ref, rtol=1e-12, atol=1e-13)
    y = O.expert_down(h, w2[0])
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-13)
    # E=1, K=1 layer = dense FFN on every token, weight exactly 1
    wg = bf16(rng.standard_normal((1, D)))
    res = O.layer(x, wg, None, w1, w3 if act == O.ACT_SWIGLU else None, w2, 1,
                  O.SOFTMAX_TOPK, act)
    assert np.all(res["w"] == 1.0)
    np.testing.assert_allclose(res["out"], y_ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("act", [O.ACT_SILU, O.ACT_SWIGLU])
@pytest.mark.parametrize("counts", [(0, 3, 5, 0, 1, 7), (4, 0, 0, 2, 9, 0), (1, 1, 1, 1, 1, 1)])
def test_grouped_ffn_uses_each_experts_own_weights(act, counts):
    # [Z] 第二层 范式 A Step 2: each expert's contiguous segment of x_perm
    # goes through that expert's own FFN.  Distinct experts, ragged
    # segments (empty first, middle and last experts) and D != Dff, checked
    # against numpy fp64 matmuls per segment: taking expert 0's weights, a
    # wrong per-expert stride or a mis-skipped empty segment all fail here.
    rng = np.random.default_rng(sum(counts) * 7 + act)
    E, D, Dff = len(counts), 64, 96
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(off[-1])
    x_perm = bf16(rng.standard_normal((rows, D)))
    w1 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w3 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w2 = bf16(rng.standard_normal((E, D, Dff)) / 10)
    h, y = O.grouped_ffn(x_perm, off, w1, w3 if act == O.ACT_SWIGLU else None, w2, act, keep_h=True)
    assert h.shape == (rows, Dff) and y.shape == (rows, D)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        h_ref, y_ref = _dense_ffn(x_perm[a:b], w1[e], w3[e], w2[e], act)
        np.testing.assert_allclose(h[a:b], h_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(y[a:b], y_ref, rtol=1e-12, atol=1e-13)
        # and not any other expert's FFN (the experts are distinct)
        other = (e + 1) % E
        _, y_other = _dense_ffn(x_perm[a:b], w1[other], w3[other], w2[other], act)
        assert np.abs(y[a:b] - y_other).max() > 1e-3


@pytest.mark.parametrize("mode", [O.SOFTMAX_TOPK, O.SIGMOID_NORM])
def test_layer_with_distinct_experts_is_the_weighted_sum_of_dense_ffns(mode):
    # [Z] 第二层 起手 dataflow: out[t] = sum_k w[t,k] FFN_{id[t,k]}(x[t]),
    # built here token by token with numpy matmuls, without any permutation
    rng = np.random.default_rng(41 + mode)
    N, D, E, K, Dff = 24, 64, 5, 2, 96
    x = bf16(rng.standard_normal((N, D)))
    wg = bf16(rng.standard_normal((E, D)) / 8)
    w1 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w3 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w2 = bf16(rng.standard_normal((E, D, Dff)) / 10)
    res = O.layer(x, wg, None, w1, w3, w2, K, mode, O.ACT_SWIGLU)
    dense = [_dense_ffn(x, w1[e], w3[e], w2[e], O.ACT_SWIGLU)[1] for e in range(E)]
    ref = np.zeros((N, D))
    for t in range(N):
        for k in range(K):
            ref[t] += res["w"][t, k] * dense[res["ids"][t, k]][t]
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-12)
    assert len(np.unique(res["ids"])) > 2      # several experts really took part


def test_silu_closed_forms():
    D, Dff = 64, 64
    x = np.zeros((1, D), np.float32); x[0, 0] = 1.0
    w1 = np.zeros((Dff, D), np.float32)
    w1[1, 0] = 1.0      # g = 1  -> silu = 1/(1+e^-1)
    w1[2, 0] = 40.0     # g = 40 -> silu ~ 40
    w1[3, 0] = -2.0     # g = -2 -> -2/(1+e^2)
    h = O.expert_up(bf16(x), bf16(w1), None, O.ACT_SILU)
    assert h[0, 0] == 0.0                      # silu(0) = 0
    assert h[0, 1] == pytest.approx(0.7310585786300049, abs=1e-16)
    assert h[0, 2] == pytest.approx(40.0, rel=1e-15)
    assert h[0, 3] == pytest.approx(-2.0 / (1.0 + math.exp(2.0)), abs=1e-16)
    w3 = np.zeros((Dff, D), np.float32); w3[:, 0] = 3.0   # u = 3 everywhere
    hs = O.expert_up(bf16(x), bf16(w1), bf16(w3), O.ACT_SWIGLU)
    np.testing.assert_allclose(hs, 3.0 * h, rtol=1e-15, atol=0)


def test_down_bf16_equals_down_on_exact_values():
    rng = np.random.default_rng(2)
    hb = bf16(rng.standard_normal((5, 64)))
    w2 = bf16(rng.standard_normal((32, 64)) / 8)
    assert np.array_equal(O.expert_down(hb, w2), O.expert_down(f64(hb), w2))


# ---------------------------------------------------------------- O7 + whole layer
@pytest.mark.parametrize("mode", [O.SOFTMAX_TOPK, O.SIGMOID_NORM])
def test_identical_experts_make_output_routing_independent(mode):
    rng = np.random.default_rng(23)
    N, D, E, K, Dff = 40, 64, 6, 3, 128
    x = bf16(rng.standard_normal((N, D)))
    wg = bf16(rng.standard_normal((E, D)) / 8)
    w1 = np.repeat(bf16(rng.standard_normal((1, Dff, D)) / 8), E, 0)
    w3 = np.repeat(bf16(rng.standard_normal((1, Dff, D)) / 8), E, 0)
    w2 = np.repeat(bf16(rng.standard_normal((1, D, Dff)) / 11), E, 0)
    res = O.layer(x, wg, None, w1, w3, w2, K, mode, O.ACT_SWIGLU)
    _, y_ref = _dense_ffn(x, w1[0], w3[0], w2[0], O.ACT_SWIGLU)
    np.testing.assert_allclose(res["out"], y_ref, rtol=1e-12, atol=1e-12)


def test_identity_experts_give_back_the_tokens():
    rng = np.random.default_rng(29)
    N, D, E, K = 50, 32, 8, 3
    x = bf16(rng.standard_normal((N, D)))
    wg = bf16(rng.standard_normal((E, D)))
    r = O.route_from_logits(O.logits(x, wg), K, O.SIGMOID_NORM)
    y = f64(O.gather_rows(x, r["perm_src"]))       # identity in place of each FFN
    out = O.combine(y, r["inv_perm"], r["w"])
    np.testing.assert_allclose(out, f64(x), rtol=1e-15, atol=1e-15)


def test_combine_weights_each_row_by_its_own_weight():
    # two tokens, two experts, rows of y distinct powers of two: the weighted
    # sum identifies exactly which row went with which weight
    y = np.array([[1.0], [2.0], [4.0], [8.0]])
    inv_perm = np.array([[0, 3], [2, 1]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    out = O.combine(y, inv_perm, w)
    assert out.tolist() == [[0.25 * 1 + 0.75 * 8], [0.5 * 4 + 0.5 * 2]]


def test_threads_do_not_change_results():
    rng = np.random.default_rng(31)
    N, D, E, K, Dff = 33, 64, 5, 2, 64
    x = bf16(rng.standard_normal((N, D)))
    wg = bf16(rng.standard_normal((E, D)) / 8)
    w1 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w3 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w2 = bf16(rng.standard_normal((E, D, Dff)) / 8)
    a = O.layer(x, wg, None, w1, w3, w2, K, O.SOFTMAX_TOPK, O.ACT_SWIGLU, nthreads=1)
    b = O.layer(x, wg, None, w1, w3, w2, K, O.SOFTMAX_TOPK, O.ACT_SWIGLU, nthreads=7)
    for k in a:
        assert np.array_equal(a[k], b[k])


# ---------------------------------------------------------------- routing statistics
def test_routing_stats_uniform_is_a_fixed_point():
    E = 8
    off = np.arange(0, 8 * 5 + 1, 5, dtype=np.int32)           # 5 rows per expert
    ema, bias, kl = O.routing_stats(off, np.full(E, 1 / E), np.zeros(E), 0.99, 0.1)
    np.testing.assert_allclose(ema, 1 / E, rtol=0, atol=1e-16)
    np.testing.assert_allclose(bias, 0.0, atol=1e-15)            # E*f - 1 = 0
    assert abs(kl - np.log(1 + 1e-9)) < 1e-15                    # f*E = 1 for every expert


def test_routing_stats_hand_computed_step():
    # E = 4, one batch with all 10 assignments on expert 2, from a uniform EMA
    off = np.array([0, 0, 0, 10, 10], np.int32)
    ema, bias, kl = O.routing_stats(off, np.full(4, 0.25), np.zeros(4), decay=0.9, step=0.1)
    exp_ema = np.array([0.225, 0.225, 0.325, 0.225])             # 0.9*0.25 + 0.1*{0,0,1,0}
    np.testing.assert_allclose(ema, exp_ema, rtol=0, atol=1e-16)
    f = exp_ema / exp_ema.sum()                                  # sum is 1 already
    np.testing.assert_allclose(bias, 0.1 * (4 * f - 1), rtol=0, atol=1e-16)
    assert bias[2] == pytest.approx(0.1 * (4 * 0.325 - 1))       # the loaded expert's bias moves by +0.03
    assert kl == pytest.approx(sum(v * np.log(v * 4 + 1e-9) for v in f), abs=1e-15)
    # a negative step moves it the other way by the same amount
    _, bias_neg, _ = O.routing_stats(off, np.full(4, 0.25), np.zeros(4), decay=0.9, step=-0.1)
    np.testing.assert_allclose(bias_neg, -bias, rtol=0, atol=0)


def test_routing_stats_empty_batch_changes_nothing():
    off = np.zeros(5, np.int32)
    ema0 = np.array([0.1, 0.2, 0.3, 0.4])
    ema, bias, kl = O.routing_stats(off, ema0, np.ones(4))
    assert np.array_equal(ema, ema0) and np.array_equal(bias, np.ones(4)) and kl == 0.0


# ---------------------------------------------------------------- paradigm B (padded)
def test_padded_placement_reproduces_the_page_buffers():
    # the page draws the same 8-token routing in padded buffers of 8 slots:
    # expert 0 [t0, t2, t5, _, ...], expert 1 [t3, t6, _, ...]
    g = json.load(open(os.path.join(GOLDEN, "permutation_example.json")))
    ids = np.array(g["assignment"], np.int32).reshape(-1, 1)
    slot, kept = O.place_padded(ids, 3, 8)
    assert kept.tolist() == [3, 2, 3]
    for e, seg in enumerate(g["segments"]):
        for j, t in enumerate(seg):
            assert slot[t, 0] == e * 8 + j
    # capacity 2: the third token of experts 0 and 2 is dropped, in token order
    slot2, kept2 = O.place_padded(ids, 3, 2)
    assert kept2.tolist() == [2, 2, 2]
    assert slot2[5, 0] == -1 and slot2[7, 0] == -1
    assert slot2[[0, 2, 3, 6, 1, 4], 0].tolist() == [0, 1, 2, 3, 4, 5]


def test_padded_capacity_formula_and_kept_counts():
    rng = np.random.default_rng(41)
    N, E, K = 300, 16, 4
    ids = np.stack([rng.permutation(E)[:K] for _ in range(N)]).astype(np.int32)
    C = math.ceil(1.5 * N * K / E)                 # the page's capacity_per_expert
    slot, kept = O.place_padded(ids, E, C)
    counts = np.bincount(ids.ravel(), minlength=E)
    assert np.array_equal(kept, np.minimum(counts, C))
    assert (slot >= 0).sum() == kept.sum()
    used = slot[slot >= 0]
    assert len(np.unique(used)) == len(used)       # no slot used twice
    for e in range(E):                             # a block fills from its start
        assert set(used[(used >= e * C) & (used < (e + 1) * C)]) == set(range(e * C, e * C + kept[e]))


def test_paradigm_b_without_drops_equals_paradigm_a():
    rng = np.random.default_rng(43)
    N, D, E, K, Dff = 24, 64, 4, 2, 64
    x = bf16(rng.standard_normal((N, D)))
    wg = bf16(rng.standard_normal((E, D)) / 8)
    w1 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w3 = bf16(rng.standard_normal((E, Dff, D)) / 8)
    w2 = bf16(rng.standard_normal((E, D, Dff)) / 8)
    a = O.layer(x, wg, None, w1, w3, w2, K, O.SOFTMAX_TOPK, O.ACT_SWIGLU)
    b = O.layer_padded(x, wg, None, w1, w3, w2, K, O.SOFTMAX_TOPK, O.ACT_SWIGLU, C=N)  # C >= any count
    assert (b["slot"] >= 0).all()
    assert np.array_equal(a["out"], b["out"])      # same rows, same arithmetic
    # and dropping removes exactly the dropped terms
    c = O.layer_padded(x, wg, None, w1, w3, w2, K, O.SOFTMAX_TOPK, O.ACT_SWIGLU, C=5)
    drop = c["slot"] < 0
    assert drop.any()
    y_a = O.grouped_ffn(O.gather_rows(x, a["perm_src"]), a["offsets"], w1, w3, w2, O.ACT_SWIGLU)
    manual = np.zeros((N, D))
    for t in range(N):
        for k in range(K):
            if not drop[t, k]:
                manual[t] += a["w"][t, k] * y_a[a["inv_perm"][t, k]]
    np.testing.assert_allclose(c["out"], manual, rtol=0, atol=1e-14)
