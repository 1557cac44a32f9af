"""fp64 CPU oracle of one MoE layer -- Python wrapper around moe_oracle.c.

TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers; the GPU product path never imports this
module and shares no code with it.

Each function marshals numpy arrays into the C oracle; the arithmetic lives in
``moe_oracle.c`` and is the plain definition of each step of the layer from
"MoE 推理完整机制：从 Router 到 Expert Parallelism 的一切" (zoe.im), sections
第一层 (router, top-K, softmax over the K selected, sigmoid + renormalise) and
第二层 范式 A Steps 1-3 (contiguous permutation with expert_offsets, per-expert
two-GEMM FFN, un-permute with router weights).

bf16 arrays are passed as numpy ``uint16`` holding the raw bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "liboracle.so")

SOFTMAX_TOPK = 0
SIGMOID_NORM = 1
ACT_SILU = 0
ACT_SWIGLU = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/liboracle.so (portable C11)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_default_threads.restype = ci
        lib.oracle_logits.argtypes = [p, p, p, i64, i64, i64, p, ci]
        lib.oracle_select.restype = ci
        lib.oracle_select.argtypes = [p, i64, i64, i64, p]
        lib.oracle_weights.argtypes = [p, p, i64, i64, i64, ci, p]
        lib.oracle_offsets.restype = ci
        lib.oracle_offsets.argtypes = [p, i64, i64, i64, p]
        lib.oracle_place.restype = ci
        lib.oracle_place.argtypes = [p, p, i64, i64, i64, p, p]
        lib.oracle_gather_rows.argtypes = [p, p, i64, i64, p]
        lib.oracle_expert_up.argtypes = [p, i64, p, p, i64, i64, ci, p, ci]
        lib.oracle_expert_down.argtypes = [p, i64, p, i64, i64, p, ci]
        lib.oracle_expert_down_bf16.argtypes = [p, i64, p, i64, i64, p, ci]
        lib.oracle_grouped_ffn.argtypes = [p, p, i64, p, p, p, i64, i64, ci, p, p, ci]
        lib.oracle_combine.argtypes = [p, p, p, i64, i64, i64, p]
        lib.oracle_place_padded.restype = ci
        lib.oracle_place_padded.argtypes = [p, i64, i64, i64, i64, p, p]
        lib.oracle_combine_kept.argtypes = [p, p, p, i64, i64, i64, p]
        lib.oracle_routing_stats.restype = ctypes.c_double
        lib.oracle_routing_stats.argtypes = [p, i64, ctypes.c_double, ctypes.c_double, p, p]
        lib.oracle_layer.restype = ci
        lib.oracle_layer.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                     ci, ci, p, p, p, p, p, p, p, ci]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode_array.argtypes = [p, i64, p]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_scale_exp.restype = ci
        lib.oracle_e4m3_scale_exp.argtypes = [ctypes.c_double]
        lib.oracle_quant_rows_e4m3.argtypes = [p, i64, i64, p, p, ci]
        lib.oracle_dequant_rows_e4m3.argtypes = [p, p, i64, i64, p]
        lib.oracle_expert_up_e4m3.argtypes = [p, p, i64, p, p, p, p, i64, i64, ci, p, ci]
        lib.oracle_expert_down_e4m3.argtypes = [p, p, i64, p, p, i64, i64, p, ci]
        lib.oracle_grouped_ffn_e4m3.argtypes = [p, p, p, i64, p, p, p, p, p, p, i64, i64, ci,
                                                p, p, p, p, p, ci]
        lib.oracle_layer_e4m3.restype = ci
        lib.oracle_layer_e4m3.argtypes = [p, p, p, p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                          ci, ci, p, p, p, p, p, p, p, ci]
        _lib = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> float64 (the bits are the top half of a binary32)."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# steps O1..O7
# --------------------------------------------------------------------------
def logits(x, wg, bias=None, nthreads: int = 0) -> np.ndarray:
    """O1: L = x Wg^T (+ bias), fp64.  x [N,D], wg [E,D] bf16 bits."""
    x = _c(x, np.uint16)
    wg = _c(wg, np.uint16)
    N, D = x.shape
    E = wg.shape[0]
    assert wg.shape[1] == D
    b = None if bias is None else _c(bias, np.float64)
    L = np.empty((N, E), np.float64)
    _load().oracle_logits(_ptr(x), _ptr(wg), _ptr(b), N, D, E, _ptr(L), nthreads)
    return L


def select(L, K: int) -> np.ndarray:
    """O2: ids [N,K] int32, ordered by (logit desc, index asc)."""
    L = _c(L, np.float64)
    N, E = L.shape
    ids = np.empty((N, K), np.int32)
    rc = _load().oracle_select(_ptr(L), N, E, K, _ptr(ids))
    if rc != 0:
        raise ValueError("oracle_select: K must be in 1..E")
    return ids


def weights(L, ids, mode: int) -> np.ndarray:
    """O3: routing weights [N,K] fp64 over the selected logits."""
    L = _c(L, np.float64)
    ids = _c(ids, np.int32)
    N, E = L.shape
    K = ids.shape[1]
    w = np.empty((N, K), np.float64)
    _load().oracle_weights(_ptr(L), _ptr(ids), N, E, K, mode, _ptr(w))
    return w


def offsets(ids, E: int) -> np.ndarray:
    """O4: expert_offsets [E+1] int32 (exclusive prefix sum of counts)."""
    ids = _c(ids, np.int32)
    N, K = ids.shape
    off = np.empty(E + 1, np.int32)
    if _load().oracle_offsets(_ptr(ids), N, K, E, _ptr(off)) != 0:
        raise ValueError("oracle_offsets: expert id out of range")
    return off


def place(ids, off, E: int):
    """O5: stable placement -> (perm_src [N*K], inv_perm [N,K]) int32."""
    ids = _c(ids, np.int32)
    off = _c(off, np.int32)
    N, K = ids.shape
    perm_src = np.empty(N * K, np.int32)
    inv_perm = np.empty((N, K), np.int32)
    if _load().oracle_place(_ptr(ids), _ptr(off), N, K, E, _ptr(perm_src), _ptr(inv_perm)) != 0:
        raise ValueError("oracle_place: expert id out of range")
    return perm_src, inv_perm


def gather_rows(x, perm_src) -> np.ndarray:
    """x_perm[r] = x[perm_src[r]] (bit copy of bf16 rows)."""
    x = _c(x, np.uint16)
    ps = _c(perm_src, np.int32)
    rows = ps.shape[0]
    D = x.shape[1]
    out = np.empty((rows, D), np.uint16)
    _load().oracle_gather_rows(_ptr(x), _ptr(ps), rows, D, _ptr(out))
    return out


def expert_up(xrows, w1, w3, act: int, nthreads: int = 0) -> np.ndarray:
    """O6a for one expert: h = silu(W1 x) * (W3 x) or silu(W1 x), fp64 [R,Dff]."""
    xrows = _c(xrows, np.uint16)
    w1 = _c(w1, np.uint16)
    R, D = xrows.shape
    Dff = w1.shape[0]
    w3c = _c(w3, np.uint16) if (w3 is not None and act == ACT_SWIGLU) else None
    h = np.empty((R, Dff), np.float64)
    _load().oracle_expert_up(_ptr(xrows), R, _ptr(w1), _ptr(w3c), D, Dff, act, _ptr(h), nthreads)
    return h


def expert_down(h, w2, nthreads: int = 0) -> np.ndarray:
    """O6b for one expert: y = W2 h.  h fp64 [R,Dff] or bf16 bits (uint16)."""
    w2 = _c(w2, np.uint16)
    D, Dff = w2.shape
    R = h.shape[0]
    y = np.empty((R, D), np.float64)
    if h.dtype == np.uint16:
        hb = _c(h, np.uint16)
        _load().oracle_expert_down_bf16(_ptr(hb), R, _ptr(w2), D, Dff, _ptr(y), nthreads)
    else:
        hf = _c(h, np.float64)
        _load().oracle_expert_down(_ptr(hf), R, _ptr(w2), D, Dff, _ptr(y), nthreads)
    return y


def grouped_ffn(x_perm, off, w1, w3, w2, act: int, keep_h: bool = False, nthreads: int = 0):
    """O6 over all experts.  Returns y [rows,D] fp64, or (h, y) with keep_h."""
    x_perm = _c(x_perm, np.uint16)
    off = _c(off, np.int32)
    w1 = _c(w1, np.uint16)
    w2 = _c(w2, np.uint16)
    E, Dff, D = w1.shape
    w3c = _c(w3, np.uint16) if (w3 is not None and act == ACT_SWIGLU) else None
    rows = int(off[E])
    y = np.empty((rows, D), np.float64)
    h = np.empty((rows, Dff), np.float64) if keep_h else None
    _load().oracle_grouped_ffn(_ptr(x_perm), _ptr(off), E, _ptr(w1), _ptr(w3c), _ptr(w2),
                               D, Dff, act, _ptr(h), _ptr(y), nthreads)
    return (h, y) if keep_h else y


def combine(y, inv_perm, w) -> np.ndarray:
    """O7: out[t] = sum_k w[t,k] y[inv_perm[t,k]] in fp64."""
    y = _c(y, np.float64)
    inv_perm = _c(inv_perm, np.int32)
    w = _c(w, np.float64)
    N, K = inv_perm.shape
    D = y.shape[1]
    out = np.empty((N, D), np.float64)
    _load().oracle_combine(_ptr(y), _ptr(inv_perm), _ptr(w), N, D, K, _ptr(out))
    return out


def layer(x, wg, bias, w1, w3, w2, K: int, mode: int, act: int, nthreads: int = 0) -> dict:
    """O1..O7 on one set of inputs; every intermediate stays fp64."""
    x = _c(x, np.uint16)
    wg = _c(wg, np.uint16)
    w1 = _c(w1, np.uint16)
    w2 = _c(w2, np.uint16)
    N, D = x.shape
    E, Dff, _ = w1.shape
    w3c = _c(w3, np.uint16) if (w3 is not None and act == ACT_SWIGLU) else None
    b = None if bias is None else _c(bias, np.float64)
    L = np.empty((N, E), np.float64)
    ids = np.empty((N, K), np.int32)
    w = np.empty((N, K), np.float64)
    off = np.empty(E + 1, np.int32)
    perm_src = np.empty(N * K, np.int32)
    inv_perm = np.empty((N, K), np.int32)
    out = np.empty((N, D), np.float64)
    rc = _load().oracle_layer(_ptr(x), _ptr(wg), _ptr(b), _ptr(w1), _ptr(w3c), _ptr(w2),
                              N, D, E, K, Dff, mode, act, _ptr(L), _ptr(ids), _ptr(w),
                              _ptr(off), _ptr(perm_src), _ptr(inv_perm), _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle_layer: bad arguments")
    return dict(logits=L, ids=ids, w=w, offsets=off, perm_src=perm_src,
                inv_perm=inv_perm, out=out)


def route_from_logits(L, K: int, mode: int, E: int | None = None) -> dict:
    """O2..O5 on given logits (e.g. fp32 logits exported by a GPU run, promoted
    exactly to fp64): ids, weights, offsets, perm_src, inv_perm."""
    L = _c(L, np.float64)
    E = L.shape[1] if E is None else E
    ids = select(L, K)
    w = weights(L, ids, mode)
    off = offsets(ids, E)
    perm_src, inv_perm = place(ids, off, E)
    return dict(ids=ids, w=w, offsets=off, perm_src=perm_src, inv_perm=inv_perm)


def routing_stats(offsets, ema, bias=None, decay: float = 0.99, step: float = 0.1):
    """EMA of expert fractions, KL to uniform and the bias step, from one
    batch's expert_offsets.  Returns (ema, bias, kl); the inputs are copied."""
    off = _c(offsets, np.int32)
    E = off.shape[0] - 1
    ema = np.array(ema, dtype=np.float64, copy=True)
    b = None if bias is None else np.array(bias, dtype=np.float64, copy=True)
    kl = _load().oracle_routing_stats(_ptr(off), E, decay, step, _ptr(ema), _ptr(b))
    return ema, b, float(kl)


def place_padded(ids, E: int, C: int):
    """Paradigm B placement: (slot [N,K] int32 with -1 = dropped, kept [E])."""
    ids = _c(ids, np.int32)
    N, K = ids.shape
    slot = np.empty((N, K), np.int32)
    kept = np.empty(E, np.int32)
    if _load().oracle_place_padded(_ptr(ids), N, K, E, C, _ptr(slot), _ptr(kept)) != 0:
        raise ValueError("oracle_place_padded: bad id or capacity")
    return slot, kept


def combine_kept(y, slot, w) -> np.ndarray:
    """out[t] = sum over kept k of w[t,k] y[slot[t,k]] (fp64)."""
    y = _c(y, np.float64)
    slot = _c(slot, np.int32)
    w = _c(w, np.float64)
    N, K = slot.shape
    D = y.shape[1]
    out = np.empty((N, D), np.float64)
    _load().oracle_combine_kept(_ptr(y), _ptr(slot), _ptr(w), N, D, K, _ptr(out))
    return out


def padded_rows(x, slot, E: int, C: int) -> np.ndarray:
    """The padded token buffer [E*C, D]: kept rows in place, zero padding."""
    x = _c(x, np.uint16)
    N, K = slot.shape
    xp = np.zeros((E * C, x.shape[1]), np.uint16)
    for t in range(N):
        for k in range(K):
            if slot[t, k] >= 0:
                xp[slot[t, k]] = x[t]
    return xp


def layer_padded(x, wg, bias, w1, w3, w2, K: int, mode: int, act: int, C: int, nthreads: int = 0) -> dict:
    """Paradigm B layer: route (O1-O3), padded placement, FFN on every row of
    the padded buffer (zero padding), weighted sum over kept assignments."""
    x = _c(x, np.uint16)
    E, Dff, D = np.asarray(w1).shape
    L = logits(x, wg, bias, nthreads)
    ids = select(L, K)
    w = weights(L, ids, mode)
    slot, kept = place_padded(ids, E, C)
    xp = padded_rows(x, slot, E, C)
    off = np.arange(0, E * C + 1, C, dtype=np.int32) if C > 0 else np.zeros(E + 1, np.int32)
    y = grouped_ffn(xp, off, w1, w3, w2, act, nthreads=nthreads)
    out = combine_kept(y, slot, w)
    return dict(logits=L, ids=ids, w=w, slot=slot, kept=kept, x_pad=xp, y_pad=y, out=out)


# --------------------------------------------------------------------------
# FP8 (e4m3) experts: per-row power-of-two scales ("MoE 推理完整机制",
# 第四层 DeepGEMM & MegaMoE: FP8 expert weights; 第三层 DeepEP: FP8 tokens)
# --------------------------------------------------------------------------
def e4m3_decode(codes) -> np.ndarray:
    """Value of every e4m3 code (fp64; NaN for 0x7f / 0xff)."""
    lib = _load()
    table = np.array([lib.oracle_e4m3_decode(c) for c in range(256)], np.float64)
    return table[np.asarray(codes, np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Nearest e4m3 code to each value (ties to even, saturating at 448)."""
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(a), a.size, _ptr(out))
    return out


def f64_to_bf16(v) -> np.ndarray:
    """Each double rounded once to bf16 (nearest, ties to even); uint16 bits."""
    a = np.asarray(v, np.float64)
    lib = _load()
    return np.array([lib.oracle_f64_to_bf16(float(x)) for x in a.ravel()], np.uint16).reshape(a.shape)


def e4m3_scale_exp(amax: float) -> int:
    """Smallest k >= -126 with amax <= 448 * 2^k."""
    return int(_load().oracle_e4m3_scale_exp(float(amax)))


def quant_rows_e4m3(src, nthreads: int = 0):
    """Per-row e4m3 quantisation of a bf16 matrix -> (codes uint8, scale float32).
    Leading dimensions are flattened into rows."""
    src = _c(src, np.uint16)
    cols = src.shape[-1]
    rows = src.size // cols if cols else 0
    q = np.empty(src.shape, np.uint8)
    sc = np.empty(src.shape[:-1], np.float32)
    _load().oracle_quant_rows_e4m3(_ptr(src), rows, cols, _ptr(q), _ptr(sc), nthreads)
    return q, sc


def dequant_rows_e4m3(q, scale) -> np.ndarray:
    """decode(q[..., c]) * scale[...] in fp64 (exact)."""
    q = _c(q, np.uint8)
    sc = _c(scale, np.float32)
    cols = q.shape[-1]
    rows = q.size // cols if cols else 0
    out = np.empty(q.shape, np.float64)
    _load().oracle_dequant_rows_e4m3(_ptr(q), _ptr(sc), rows, cols, _ptr(out))
    return out


def expert_up_e4m3(xq, sx, w1q, s1, w3q, s3, act: int, nthreads: int = 0) -> np.ndarray:
    """FP8 first GEMM + activation for one expert's rows; fp64 [R,Dff]."""
    xq = _c(xq, np.uint8)
    sx = _c(sx, np.float32)
    w1q = _c(w1q, np.uint8)
    s1 = _c(s1, np.float32)
    R, D = xq.shape
    Dff = w1q.shape[0]
    sw = act == ACT_SWIGLU
    w3c = _c(w3q, np.uint8) if sw else None
    s3c = _c(s3, np.float32) if sw else None
    h = np.empty((R, Dff), np.float64)
    _load().oracle_expert_up_e4m3(_ptr(xq), _ptr(sx), R, _ptr(w1q), _ptr(s1), _ptr(w3c), _ptr(s3c),
                                  D, Dff, act, _ptr(h), nthreads)
    return h


def expert_down_e4m3(hq, sh, w2q, s2, nthreads: int = 0) -> np.ndarray:
    """FP8 second GEMM for one expert's rows; fp64 [R,D]."""
    hq = _c(hq, np.uint8)
    sh = _c(sh, np.float32)
    w2q = _c(w2q, np.uint8)
    s2 = _c(s2, np.float32)
    R, Dff = hq.shape
    D = w2q.shape[0]
    y = np.empty((R, D), np.float64)
    _load().oracle_expert_down_e4m3(_ptr(hq), _ptr(sh), R, _ptr(w2q), _ptr(s2), D, Dff, _ptr(y), nthreads)
    return y


def grouped_ffn_e4m3(xq_perm, sx_perm, off, w1q, s1, w3q, s3, w2q, s2, act: int, nthreads: int = 0) -> dict:
    """FP8 FFN over all experts: h (fp64), hb (bf16 of h), hq / sh (its per-row
    e4m3 quantisation) and y (fp64)."""
    xq_perm = _c(xq_perm, np.uint8)
    sx_perm = _c(sx_perm, np.float32)
    off = _c(off, np.int32)
    w1q = _c(w1q, np.uint8)
    s1 = _c(s1, np.float32)
    w2q = _c(w2q, np.uint8)
    s2 = _c(s2, np.float32)
    E, Dff, D = w1q.shape
    sw = act == ACT_SWIGLU
    w3c = _c(w3q, np.uint8) if sw else None
    s3c = _c(s3, np.float32) if sw else None
    rows = int(off[E])
    h = np.empty((rows, Dff), np.float64)
    hb = np.empty((rows, Dff), np.uint16)
    hq = np.empty((rows, Dff), np.uint8)
    sh = np.empty(rows, np.float32)
    y = np.empty((rows, D), np.float64)
    _load().oracle_grouped_ffn_e4m3(_ptr(xq_perm), _ptr(sx_perm), _ptr(off), E, _ptr(w1q), _ptr(s1),
                                    _ptr(w3c), _ptr(s3c), _ptr(w2q), _ptr(s2), D, Dff, act,
                                    _ptr(h), _ptr(hb), _ptr(hq), _ptr(sh), _ptr(y), nthreads)
    return dict(h=h, hb=hb, hq=hq, sh=sh, y=y)


def layer_e4m3(x, wg, bias, w1q, s1, w3q, s3, w2q, s2, K: int, mode: int, act: int,
               nthreads: int = 0) -> dict:
    """The layer with FP8 experts: bf16 routing (O1..O5), per-token e4m3 x,
    the FP8 FFN, the fp64 combine."""
    x = _c(x, np.uint16)
    wg = _c(wg, np.uint16)
    w1q = _c(w1q, np.uint8)
    s1 = _c(s1, np.float32)
    w2q = _c(w2q, np.uint8)
    s2 = _c(s2, np.float32)
    N, D = x.shape
    E, Dff, _ = w1q.shape
    sw = act == ACT_SWIGLU
    w3c = _c(w3q, np.uint8) if sw else None
    s3c = _c(s3, np.float32) if sw else None
    b = None if bias is None else _c(bias, np.float64)
    L = np.empty((N, E), np.float64)
    ids = np.empty((N, K), np.int32)
    w = np.empty((N, K), np.float64)
    off = np.empty(E + 1, np.int32)
    perm_src = np.empty(N * K, np.int32)
    inv_perm = np.empty((N, K), np.int32)
    out = np.empty((N, D), np.float64)
    rc = _load().oracle_layer_e4m3(_ptr(x), _ptr(wg), _ptr(b), _ptr(w1q), _ptr(s1), _ptr(w3c), _ptr(s3c),
                                   _ptr(w2q), _ptr(s2), N, D, E, K, Dff, mode, act, _ptr(L), _ptr(ids),
                                   _ptr(w), _ptr(off), _ptr(perm_src), _ptr(inv_perm), _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle_layer_e4m3: bad arguments")
    return dict(logits=L, ids=ids, w=w, offsets=off, perm_src=perm_src, inv_perm=inv_perm, out=out)
