"""Pins of the oracle's FP8 (e4m3) experts to facts outside the oracle.

The pages name FP8 expert weights ("MoE 推理完整机制：从 Router 到 Expert
Parallelism 的一切", 第四层 DeepGEMM & MegaMoE) and FP8 token hidden states
(第三层, DeepEP) without fixing a format; the reading pinned here is e4m3 codes
with one power-of-two scale per row.  The checks use routes to the answer that
do not pass through the oracle's code: the e4m3 format's definition worked by
hand, torch's float8_e4m3fn conversions (on the inputs where torch and a
saturating round-to-nearest-even agree), error bounds of the format, and
operands built so that quantisation is exact, where the FP8 GEMMs must
reproduce the independently pinned bf16 oracle bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O


def bf16_bits_of(values) -> np.ndarray:
    """bf16 bits of values that are exactly representable in bf16."""
    f = np.asarray(values, np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(O.bf16_to_f64(bits), f.astype(np.float64)), "value not exact in bf16"
    return bits


# ------------------------------------------------------------------ codec
def test_e4m3_decode_hand_values():
    # sign | exponent (bias 7) | mantissa, worked from the format definition
    cases = {
        0x00: 0.0,
        0x01: 2.0 ** -9,           # smallest subnormal: 1/8 * 2^-6
        0x07: 7 * 2.0 ** -9,       # largest subnormal
        0x08: 2.0 ** -6,           # smallest normal
        0x30: 0.5,
        0x38: 1.0,                 # exponent field 7 = bias
        0x3c: 1.5,
        0x40: 2.0,
        0x77: 240.0,               # 1.875 * 2^7
        0x7e: 448.0,               # largest finite: exponent 15, mantissa 6
        0x80: -0.0,
        0xb8: -1.0,
        0xc5: -3.25,               # -(1 + 5/8) * 2
        0xfe: -448.0,
    }
    got = O.e4m3_decode(list(cases))
    for (code, want), g in zip(cases.items(), got):
        assert g == want and np.signbit(g) == np.signbit(want), hex(code)
    assert np.isnan(O.e4m3_decode([0x7f, 0xff])).all()


def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_encode_matches_torch_on_every_bf16_value_in_range():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        v = O.bf16_to_f64(bits)
    keep = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[keep]
    # torch rounds to nearest-even and agrees with saturation inside the range
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(v)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(v[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_e4m3_encode_ties_subnormals_and_saturation():
    cases = [
        (1.0 + 1 / 16, 0x38),        # halfway 1 and 1.125 -> even mantissa (1.0)
        (1.0 + 3 / 16, 0x3a),        # halfway 1.125 and 1.25 -> even (1.25)
        (1.0 + 1 / 16 + 2 ** -30, 0x39),  # just above the tie -> up
        (2.0 ** -10, 0x00),          # half the smallest subnormal -> 0
        (3 * 2.0 ** -10, 0x02),      # halfway codes 1 and 2 -> even (2)
        (2.0 ** -10 + 2 ** -40, 0x01),
        (1.875 * 2 ** -6 + 2 ** -10, 0x10),  # tie across the subnormal/normal edge -> 0x10
        (464.0, 0x7e),               # past 448: saturate
        (480.0, 0x7e),
        (1e30, 0x7e),
        (-1e30, 0xfe),
        (-(2.0 ** -11), 0x80),       # rounds to zero, keeps the sign
        (-0.0, 0x80),
        (0.0, 0x00),
    ]
    got = O.e4m3_encode([c[0] for c in cases])
    for (v, want), g in zip(cases, got):
        assert g == want, (v, hex(g), hex(want))


def test_f64_to_bf16_matches_torch_on_float_inputs():
    rng = np.random.default_rng(5)
    f = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 3000),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, -1e-42], np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_f64_to_bf16_rounds_once_from_the_double():
    # 1 + 2^-8 is the tie between 1 and 1 + 2^-7; a hair above it must go up.
    # (Rounding through binary32 first would lose the hair and give 1.0.)
    assert O.f64_to_bf16(1 + 2 ** -8 + 2 ** -30) == 0x3f81
    assert O.f64_to_bf16(1 + 2 ** -8) == 0x3f80               # exact tie -> even
    assert O.f64_to_bf16(1 + 3 * 2 ** -8) == 0x3f82           # tie -> even (up)
    assert O.f64_to_bf16(2.0 ** -133) == 0x0001               # smallest subnormal
    assert O.f64_to_bf16(2.0 ** -134) == 0x0000               # tie with 0 -> even
    assert O.f64_to_bf16(3 * 2.0 ** -134) == 0x0002           # tie 1/2 ulps -> even
    assert O.f64_to_bf16((2 - 2 ** -7) * 2.0 ** 127) == 0x7f7f  # largest finite
    assert O.f64_to_bf16((2 - 2 ** -8) * 2.0 ** 127) == 0x7f80  # tie at the top -> inf
    assert O.f64_to_bf16(-2.5) == 0xc020


# ------------------------------------------------------------------ scales
@pytest.mark.parametrize("amax,k", [
    (448.0, 0), (448.5, 1), (449.0, 1), (896.0, 1), (896.5, 2), (224.0, -1), (224.5, 0),
    (1.0, -8),            # 448 / 256 = 1.75 >= 1 > 448 / 512
    (1.75, -8), (1.7578125, -7),
    (0.0, -126), (2.0 ** -140, -126),   # zero rows and tiny rows stop at 2^-126
    (3.0e38, 120),
])
def test_scale_exponent_hand_values(amax, k):
    assert O.e4m3_scale_exp(amax) == k


def _rows_with_spread(rng, rows, cols):
    mags = 2.0 ** rng.integers(-20, 20, size=(rows, 1))
    x = (rng.standard_normal((rows, cols)) * mags).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits


def test_quantised_rows_fill_the_top_binade_and_respect_the_error_bound():
    rng = np.random.default_rng(7)
    bits = _rows_with_spread(rng, 64, 300)
    bits[3] = 0                                    # an all-zero row
    q, sc = O.quant_rows_e4m3(bits)
    x = O.bf16_to_f64(bits)
    xq = O.dequant_rows_e4m3(q, sc)
    dec = O.e4m3_decode(q)
    for r in range(bits.shape[0]):
        amax = np.abs(x[r]).max()
        if amax == 0:
            assert sc[r] == 2.0 ** -126 and (q[r] & 0x7f).max() == 0
            continue
        # the row maximum lands in (224, 448] after scaling, never beyond
        m = np.abs(dec[r]).max()
        assert 224.0 <= m <= 448.0
        assert amax / sc[r] <= 448.0 and amax / sc[r] > 224.0
        # power-of-two scale
        assert np.frexp(sc[r])[0] == 0.5
    # error: at most half a unit in the last place of e4m3 (normals: 2^-4
    # relative; subnormals: 2^-10 in scaled units)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, sc[:, None].astype(np.float64) * 2.0 ** -10)
    assert (np.abs(xq - x) <= bound).all()


def test_representable_rows_round_trip_exactly():
    rng = np.random.default_rng(11)
    rows, cols = 32, 96
    codes = rng.integers(0, 127, size=(rows, cols)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=(rows, cols)) << 7).astype(np.uint8)
    codes[:, 0] = 0x7e                                # row max 448 fixes the scale
    k = rng.integers(-30, 30, size=rows)
    vals = O.e4m3_decode(codes) * (2.0 ** k)[:, None]
    bits = bf16_bits_of(vals)
    q, sc = O.quant_rows_e4m3(bits)
    assert np.array_equal(sc, (2.0 ** k).astype(np.float32))
    # equal values, and equal codes up to the sign of zero
    assert np.array_equal(O.e4m3_decode(q), O.e4m3_decode(codes))


# ------------------------------------------------------------------ GEMMs
def _representable_matrix(rng, rows, cols):
    """bf16 bits of a matrix whose per-row quantisation is exact."""
    codes = rng.integers(0, 0x7e, size=(rows, cols)).astype(np.uint8)
    codes |= (rng.integers(0, 2, size=(rows, cols)) << 7).astype(np.uint8)
    codes[np.arange(rows), rng.integers(0, cols, rows)] = 0x70  # 256: row max in (224, 448]
    codes[:, :] = np.where((codes & 0x7f) > 0x70, codes & 0x80 | 0x70, codes)
    k = rng.integers(-12, -4, size=rows)
    return bf16_bits_of(O.e4m3_decode(codes) * (2.0 ** k)[:, None])


@pytest.mark.parametrize("act", [O.ACT_SWIGLU, O.ACT_SILU])
def test_fp8_gemms_equal_the_bf16_oracle_on_representable_operands(act):
    rng = np.random.default_rng(13)
    R, D, Dff = 5, 64, 48
    x = _representable_matrix(rng, R, D)
    w1 = _representable_matrix(rng, Dff, D)
    w3 = _representable_matrix(rng, Dff, D)
    w2 = _representable_matrix(rng, D, Dff)
    xq, sx = O.quant_rows_e4m3(x)
    w1q, s1 = O.quant_rows_e4m3(w1)
    w3q, s3 = O.quant_rows_e4m3(w3)
    w2q, s2 = O.quant_rows_e4m3(w2)
    h8 = O.expert_up_e4m3(xq, sx, w1q, s1, w3q, s3, act)
    h16 = O.expert_up(x, w1, w3, act)
    assert np.array_equal(h8, h16)
    hb = _representable_matrix(rng, R, Dff)
    hq, sh = O.quant_rows_e4m3(hb)
    assert np.array_equal(O.expert_down_e4m3(hq, sh, w2q, s2), O.expert_down(hb, w2))


def test_grouped_fp8_ffn_is_its_steps_in_order():
    rng = np.random.default_rng(17)
    E, D, Dff = 3, 64, 32
    off = np.array([0, 4, 4, 9], np.int32)            # one empty expert
    x = torch.randn(9, D).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w1 = (torch.randn(E, Dff, D) / 8).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w3 = (torch.randn(E, Dff, D) / 8).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w2 = (torch.randn(E, D, Dff) / 6).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xq, sx = O.quant_rows_e4m3(x)
    w1q, s1 = O.quant_rows_e4m3(w1)
    w3q, s3 = O.quant_rows_e4m3(w3)
    w2q, s2 = O.quant_rows_e4m3(w2)
    g = O.grouped_ffn_e4m3(xq, sx, off, w1q, s1, w3q, s3, w2q, s2, O.ACT_SWIGLU)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        h = O.expert_up_e4m3(xq[a:b], sx[a:b], w1q[e], s1[e], w3q[e], s3[e], O.ACT_SWIGLU)
        assert np.array_equal(g["h"][a:b], h)
    assert np.array_equal(g["hb"], O.f64_to_bf16(g["h"]))
    hq, sh = O.quant_rows_e4m3(g["hb"])
    assert np.array_equal(g["hq"], hq) and np.array_equal(g["sh"], sh)
    for e in range(E):
        a, b = off[e], off[e + 1]
        if a < b:
            assert np.array_equal(g["y"][a:b], O.expert_down_e4m3(hq[a:b], sh[a:b], w2q[e], s2[e]))
    _ = rng


def test_fp8_layer_routes_like_the_bf16_layer_and_stays_close_to_it():
    torch.manual_seed(3)
    N, D, E, K, Dff = 40, 128, 8, 2, 64
    def b(t):
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    x = b(torch.randn(N, D))
    wg = b(torch.randn(E, D) / D ** 0.5)
    w1 = b(torch.randn(E, Dff, D) / D ** 0.5)
    w3 = b(torch.randn(E, Dff, D) / D ** 0.5)
    w2 = b(torch.randn(E, D, Dff) / Dff ** 0.5)
    ref = O.layer(x, wg, None, w1, w3, w2, K, O.SOFTMAX_TOPK, O.ACT_SWIGLU)
    w1q, s1 = O.quant_rows_e4m3(w1)
    w3q, s3 = O.quant_rows_e4m3(w3)
    w2q, s2 = O.quant_rows_e4m3(w2)
    got = O.layer_e4m3(x, wg, None, w1q, s1, w3q, s3, w2q, s2, K, O.SOFTMAX_TOPK, O.ACT_SWIGLU)
    for key in ("ids", "offsets", "perm_src", "inv_perm"):
        assert np.array_equal(got[key], ref[key])
    assert np.array_equal(got["w"], ref["w"])
    # the layer is the composition of its steps
    xq, sx = O.quant_rows_e4m3(x)
    ps = got["perm_src"]
    g = O.grouped_ffn_e4m3(xq[ps], sx[ps], got["offsets"], w1q, s1, w3q, s3, w2q, s2, O.ACT_SWIGLU)
    assert np.array_equal(got["out"], O.combine(g["y"], got["inv_perm"], got["w"]))
    # three e4m3 roundings per path: within a few percent of the exact layer
    err = np.linalg.norm(got["out"] - ref["out"]) / np.linalg.norm(ref["out"])
    assert 1e-3 < err < 0.1, err
