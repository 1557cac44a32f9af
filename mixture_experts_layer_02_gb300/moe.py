"""Thin Python binding of libmoe.so (include/moe.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no
fallback: if libmoe.so is missing or cannot load, every call raises.

Functions carry the C names (``moe_route``, ``moe_permute``,
``moe_grouped_ffn``, ``moe_combine``, ``moe_layer_forward``) and take torch
tensors that already live on the current CUDA device.  Outputs not passed in
are allocated here with torch.  ``ws`` is a workspace tensor from
:func:`workspace`; pass the same one again to avoid re-allocating.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_BOUNDS = 5
MOE_ERR_DEVICE_TIMEOUT = 6

SOFTMAX_TOPK = 0
SIGMOID_NORM = 1
ACT_SILU = 0
ACT_SWIGLU = 1

EXPORTED = (
    "moe_workspace_size", "moe_route", "moe_permute", "moe_route_permute", "moe_grouped_ffn", "moe_combine",
    "moe_layer_forward", "moe_layer_workspace_layout", "moe_read_device_error",
    "moe_clear_device_error", "moe_set_debug_flags", "moe_status_string",
    "moe_last_error_detail", "moe_version", "moe_permute_static_scratch", "moe_routing_stats",
    "moe_capacity", "moe_workspace_size_padded", "moe_permute_padded", "moe_combine_padded",
    "moe_layer_forward_padded", "moe_layer_padded_workspace_layout", "moe_layer_launches",
    "moe_quantize_e4m3", "moe_permute_e4m3", "moe_grouped_ffn_e4m3", "moe_layer_forward_e4m3",
    "moe_layer_e4m3_workspace_layout", "moe_layer_launches_e4m3", "moe_permute_indices",
    "moe_grouped_ffn_gathered", "moe_grouped_ffn_e4m3_gathered",
)

_lock = threading.Lock()
_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        super().__init__(f"{fn} failed: status {status} ({status_string(status)}): {detail}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so and declare every exported signature."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libmoe.so not found at {path}: build it with "
                               "`python -m mixture_experts_layer_02_gb300.build`")
        L = ctypes.CDLL(path)
        p, i, sz, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint32
        L.moe_workspace_size.restype = sz
        L.moe_workspace_size.argtypes = [ctypes.c_char_p, i, i, i, i, i]
        L.moe_route.restype = i
        L.moe_route.argtypes = [p, p, p, i, i, i, i, i, p, p, p, p, sz, p]
        L.moe_permute.restype = i
        L.moe_permute.argtypes = [p, p, i, i, i, i, p, p, p, p, p, sz, p]
        L.moe_route_permute.restype = i
        L.moe_route_permute.argtypes = [p, p, p, i, i, i, i, i, p, p, p, p, p, p, p, sz, p]
        L.moe_permute_static_scratch.restype = i
        L.moe_permute_static_scratch.argtypes = [p, p, i, i, i, i, p, p, p, p, p]
        L.moe_grouped_ffn.restype = i
        L.moe_grouped_ffn.argtypes = [p, p, i, p, p, p, i, i, i, i, p, p, p, sz, p]
        L.moe_combine.restype = i
        L.moe_combine.argtypes = [p, p, p, i, i, i, p, p, sz, p]
        L.moe_layer_forward.restype = i
        L.moe_layer_forward.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, p, p, sz, p]
        L.moe_layer_launches.restype = i
        L.moe_layer_launches.argtypes = [i, i, i, i, i, i, i]
        L.moe_capacity.restype = i
        L.moe_capacity.argtypes = [i, i, i, ctypes.c_float]
        L.moe_workspace_size_padded.restype = sz
        L.moe_workspace_size_padded.argtypes = [ctypes.c_char_p, i, i, i, i, i, i]
        L.moe_permute_padded.restype = i
        L.moe_permute_padded.argtypes = [p, p, i, i, i, i, i, p, p, p, p, p, sz, p]
        L.moe_combine_padded.restype = i
        L.moe_combine_padded.argtypes = [p, p, p, i, i, i, i, i, p, p, sz, p]
        L.moe_layer_forward_padded.restype = i
        L.moe_layer_forward_padded.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, i, i, p, p, sz, p]
        L.moe_layer_padded_workspace_layout.restype = i
        L.moe_layer_padded_workspace_layout.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_routing_stats.restype = i
        L.moe_routing_stats.argtypes = [p, i, ctypes.c_float, ctypes.c_float, p, p, p, p]
        L.moe_layer_workspace_layout.restype = i
        L.moe_layer_workspace_layout.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_quantize_e4m3.restype = i
        L.moe_quantize_e4m3.argtypes = [p, ctypes.c_longlong, i, p, p, p]
        L.moe_permute_e4m3.restype = i
        L.moe_permute_e4m3.argtypes = [p, p, i, i, i, i, p, p, p, p, p, sz, p]
        L.moe_grouped_ffn_e4m3.restype = i
        L.moe_grouped_ffn_e4m3.argtypes = [p, p, p, p, i, p, p, p, p, p, p, i, i, i, i, p, p, p, p, p, sz, p]
        L.moe_layer_forward_e4m3.restype = i
        L.moe_layer_forward_e4m3.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, i, i, p, p, sz, p]
        L.moe_layer_e4m3_workspace_layout.restype = i
        L.moe_layer_e4m3_workspace_layout.argtypes = [i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_layer_launches_e4m3.restype = i
        L.moe_layer_launches_e4m3.argtypes = [i, i, i, i, i, i]
        L.moe_permute_indices.restype = i
        L.moe_permute_indices.argtypes = [p, i, i, i, p, p, p, p, sz, p]
        L.moe_grouped_ffn_gathered.restype = i
        L.moe_grouped_ffn_gathered.argtypes = [p, i, p, p, i, p, p, p, i, i, i, i, p, p, p, sz, p]
        L.moe_grouped_ffn_e4m3_gathered.restype = i
        L.moe_grouped_ffn_e4m3_gathered.argtypes = [p, p, i, p, p, i, p, p, p, p, p, p, i, i, i, i,
                                                    p, p, p, p, p, sz, p]
        L.moe_read_device_error.restype = i
        L.moe_read_device_error.argtypes = [p, p]
        L.moe_clear_device_error.restype = i
        L.moe_clear_device_error.argtypes = [p, p]
        L.moe_set_debug_flags.restype = i
        L.moe_set_debug_flags.argtypes = [p, u32, p]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i]
        L.moe_last_error_detail.restype = ctypes.c_char_p
        L.moe_last_error_detail.argtypes = []
        L.moe_version.restype = ctypes.c_char_p
        L.moe_version.argtypes = []
        _lib = L
        return L


def status_string(s: int) -> str:
    return load().moe_status_string(s).decode()


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status, load().moe_last_error_detail().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")


# ---------------------------------------------------------------- workspace
def workspace_size(op: str, N=0, D=0, E=0, K=0, Dff=0) -> int:
    return int(load().moe_workspace_size(op.encode(), N, D, E, K, Dff))


def workspace(op: str, N=0, D=0, E=0, K=0, Dff=0, device=None) -> torch.Tensor:
    """A zero-initialised workspace tensor (uint8) for ``op``."""
    n = workspace_size(op, N, D, E, K, Dff)
    if n == 0:
        raise ValueError(f"invalid workspace request {op} N={N} D={D} E={E} K={K} Dff={Dff}")
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def layer_launches(N, D, E, K, Dff, act, cap=-1) -> int:
    """Kernels one layer call launches (cap >= 0: the padded paradigm)."""
    return int(load().moe_layer_launches(N, D, E, K, Dff, act, cap))


def layer_workspace_layout(N, D, E, K, Dff) -> list:
    arr = (ctypes.c_size_t * 8)()
    if load().moe_layer_workspace_layout(N, D, E, K, Dff, arr) != 0:
        raise ValueError("invalid sizes")
    return list(arr)


def read_device_error(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the workspace's device status."""
    return int(load().moe_read_device_error(_ptr(ws), _stream(stream)))


def clear_device_error(ws: torch.Tensor, stream=None):
    _check("moe_clear_device_error", load().moe_clear_device_error(_ptr(ws), _stream(stream)))


def set_debug_flags(ws: torch.Tensor, flags: int, stream=None):
    _check("moe_set_debug_flags", load().moe_set_debug_flags(_ptr(ws), flags, _stream(stream)))


# ---------------------------------------------------------------- entry points
def moe_route(x, w_gate, bias, K: int, mode: int, topk_ids=None, topk_w=None,
              logits_out=None, ws=None, stream=None):
    N, D = x.shape
    E = w_gate.shape[0]
    _need(x, torch.bfloat16, (N, D), "x")
    _need(w_gate, torch.bfloat16, (E, D), "w_gate")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    dev = x.device
    topk_ids = torch.empty((N, K), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    topk_w = torch.empty((N, K), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    _need(topk_ids, torch.int32, (N, K), "topk_ids")
    _need(topk_w, torch.float32, (N, K), "topk_w")
    if logits_out is not None:
        _need(logits_out, torch.float32, (N, E), "logits_out")
    ws = workspace("route", N, D, E, K, device=dev) if ws is None else ws
    _check("moe_route", load().moe_route(
        _ptr(x), _ptr(w_gate), _ptr(bias), N, D, E, K, mode, _ptr(topk_ids), _ptr(topk_w),
        _ptr(logits_out), _ptr(ws), ws.numel(), _stream(stream)))
    return topk_ids, topk_w


def moe_permute(x, topk_ids, E: int, expert_offsets=None, perm_src=None, inv_perm=None,
                x_perm=None, ws=None, stream=None):
    N, D = x.shape
    K = topk_ids.shape[1]
    _need(x, torch.bfloat16, (N, D), "x")
    _need(topk_ids, torch.int32, (N, K), "topk_ids")
    dev = x.device
    expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if expert_offsets is None else expert_offsets
    perm_src = torch.empty(N * K, dtype=torch.int32, device=dev) if perm_src is None else perm_src
    inv_perm = torch.empty((N, K), dtype=torch.int32, device=dev) if inv_perm is None else inv_perm
    x_perm = torch.empty((N * K, D), dtype=torch.bfloat16, device=dev) if x_perm is None else x_perm
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _need(perm_src, torch.int32, (N * K,), "perm_src")
    _need(inv_perm, torch.int32, (N, K), "inv_perm")
    _need(x_perm, torch.bfloat16, (N * K, D), "x_perm")
    ws = workspace("permute", N=N, E=E, device=dev) if ws is None else ws
    _check("moe_permute", load().moe_permute(
        _ptr(x), _ptr(topk_ids), N, D, E, K, _ptr(expert_offsets), _ptr(perm_src),
        _ptr(inv_perm), _ptr(x_perm), _ptr(ws), ws.numel(), _stream(stream)))
    return expert_offsets, perm_src, inv_perm, x_perm


def moe_route_permute(x, w_gate, bias, K: int, mode: int, topk_ids=None, topk_w=None, expert_offsets=None,
                      perm_src=None, inv_perm=None, x_perm=None, ws=None, stream=None):
    """moe_route then moe_permute as one call; decode-sized calls (up to 8
    tokens, N*K <= 256) select and permute in one launch.  Returns (topk_ids, topk_w,
    expert_offsets, perm_src, inv_perm, x_perm)."""
    N, D = x.shape
    E = w_gate.shape[0]
    _need(x, torch.bfloat16, (N, D), "x")
    _need(w_gate, torch.bfloat16, (E, D), "w_gate")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    dev = x.device
    topk_ids = torch.empty((N, K), dtype=torch.int32, device=dev) if topk_ids is None else topk_ids
    topk_w = torch.empty((N, K), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if expert_offsets is None else expert_offsets
    perm_src = torch.empty(N * K, dtype=torch.int32, device=dev) if perm_src is None else perm_src
    inv_perm = torch.empty((N, K), dtype=torch.int32, device=dev) if inv_perm is None else inv_perm
    x_perm = torch.empty((N * K, D), dtype=torch.bfloat16, device=dev) if x_perm is None else x_perm
    _need(topk_ids, torch.int32, (N, K), "topk_ids")
    _need(topk_w, torch.float32, (N, K), "topk_w")
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _need(perm_src, torch.int32, (N * K,), "perm_src")
    _need(inv_perm, torch.int32, (N, K), "inv_perm")
    _need(x_perm, torch.bfloat16, (N * K, D), "x_perm")
    ws = workspace("route_permute", N, D, E, K, device=dev) if ws is None else ws
    _check("moe_route_permute", load().moe_route_permute(
        _ptr(x), _ptr(w_gate), _ptr(bias), N, D, E, K, mode, _ptr(topk_ids), _ptr(topk_w), _ptr(expert_offsets),
        _ptr(perm_src), _ptr(inv_perm), _ptr(x_perm), _ptr(ws), ws.numel(), _stream(stream)))
    return topk_ids, topk_w, expert_offsets, perm_src, inv_perm, x_perm


def moe_permute_static_scratch(x, topk_ids, E: int, expert_offsets=None, perm_src=None,
                               inv_perm=None, x_perm=None, stream=None):
    """moe_permute for callers that cannot allocate: the scratch is a fixed
    4 MiB array inside the library (see include/moe.h); no workspace."""
    N, D = x.shape
    K = topk_ids.shape[1]
    _need(x, torch.bfloat16, (N, D), "x")
    _need(topk_ids, torch.int32, (N, K), "topk_ids")
    dev = x.device
    expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if expert_offsets is None else expert_offsets
    perm_src = torch.empty(N * K, dtype=torch.int32, device=dev) if perm_src is None else perm_src
    inv_perm = torch.empty((N, K), dtype=torch.int32, device=dev) if inv_perm is None else inv_perm
    x_perm = torch.empty((N * K, D), dtype=torch.bfloat16, device=dev) if x_perm is None else x_perm
    _check("moe_permute_static_scratch", load().moe_permute_static_scratch(
        _ptr(x), _ptr(topk_ids), N, D, E, K, _ptr(expert_offsets), _ptr(perm_src),
        _ptr(inv_perm), _ptr(x_perm), _stream(stream)))
    return expert_offsets, perm_src, inv_perm, x_perm


def moe_grouped_ffn(x_perm, expert_offsets, w1, w3, w2, act: int, h=None, y_perm=None,
                    ws=None, stream=None):
    rows, D = x_perm.shape
    E, Dff, _ = w1.shape
    _need(x_perm, torch.bfloat16, (rows, D), "x_perm")
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _need(w1, torch.bfloat16, (E, Dff, D), "w1")
    if act == ACT_SWIGLU:
        _need(w3, torch.bfloat16, (E, Dff, D), "w3")
    _need(w2, torch.bfloat16, (E, D, Dff), "w2")
    dev = x_perm.device
    h = torch.empty((rows, Dff), dtype=torch.bfloat16, device=dev) if h is None else h
    y_perm = torch.empty((rows, D), dtype=torch.bfloat16, device=dev) if y_perm is None else y_perm
    _need(h, torch.bfloat16, (rows, Dff), "h")
    _need(y_perm, torch.bfloat16, (rows, D), "y_perm")
    ws = workspace("ffn", rows, D, E, 1, Dff, device=dev) if ws is None else ws
    _check("moe_grouped_ffn", load().moe_grouped_ffn(
        _ptr(x_perm), _ptr(expert_offsets), rows, _ptr(w1),
        _ptr(w3) if act == ACT_SWIGLU else None, _ptr(w2), E, D, Dff, act, _ptr(h),
        _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))
    return h, y_perm


def moe_permute_indices(topk_ids, E: int, expert_offsets=None, perm_src=None, inv_perm=None, ws=None,
                        stream=None):
    """The permutation's indices without the row copy (for the gathered FFN)."""
    N, K = topk_ids.shape
    _need(topk_ids, torch.int32, (N, K), "topk_ids")
    dev = topk_ids.device
    expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if expert_offsets is None else expert_offsets
    perm_src = torch.empty(N * K, dtype=torch.int32, device=dev) if perm_src is None else perm_src
    inv_perm = torch.empty((N, K), dtype=torch.int32, device=dev) if inv_perm is None else inv_perm
    ws = workspace("permute", N=N, E=E, device=dev) if ws is None else ws
    _check("moe_permute_indices", load().moe_permute_indices(
        _ptr(topk_ids), N, E, K, _ptr(expert_offsets), _ptr(perm_src), _ptr(inv_perm), _ptr(ws), ws.numel(),
        _stream(stream)))
    return expert_offsets, perm_src, inv_perm


def moe_grouped_ffn_gathered(x, perm_src, expert_offsets, w1, w3, w2, act: int, h=None, y_perm=None,
                             ws=None, stream=None):
    """moe_grouped_ffn with GEMM1 reading token rows of x through perm_src."""
    N, D = x.shape
    rows = perm_src.shape[0]
    E, Dff, _ = w1.shape
    _need(x, torch.bfloat16, (N, D), "x")
    _need(perm_src, torch.int32, (rows,), "perm_src")
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    dev = x.device
    h = torch.empty((rows, Dff), dtype=torch.bfloat16, device=dev) if h is None else h
    y_perm = torch.empty((rows, D), dtype=torch.bfloat16, device=dev) if y_perm is None else y_perm
    ws = workspace("ffn", rows, D, E, 1, Dff, device=dev) if ws is None else ws
    _check("moe_grouped_ffn_gathered", load().moe_grouped_ffn_gathered(
        _ptr(x), N, _ptr(perm_src), _ptr(expert_offsets), rows, _ptr(w1),
        _ptr(w3) if act == ACT_SWIGLU else None, _ptr(w2), E, D, Dff, act, _ptr(h), _ptr(y_perm),
        _ptr(ws), ws.numel(), _stream(stream)))
    return h, y_perm


def moe_combine(y_perm, inv_perm, topk_w, out=None, ws=None, stream=None):
    N, K = inv_perm.shape
    D = y_perm.shape[1]
    _need(y_perm, torch.bfloat16, (N * K, D), "y_perm")
    _need(inv_perm, torch.int32, (N, K), "inv_perm")
    _need(topk_w, torch.float32, (N, K), "topk_w")
    dev = y_perm.device
    out = torch.empty((N, D), dtype=torch.bfloat16, device=dev) if out is None else out
    _need(out, torch.bfloat16, (N, D), "out")
    ws = workspace("combine", device=dev) if ws is None else ws
    _check("moe_combine", load().moe_combine(
        _ptr(y_perm), _ptr(inv_perm), _ptr(topk_w), N, D, K, _ptr(out), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def moe_layer_forward(x, w_gate, bias, w1, w3, w2, K: int, mode: int, act: int, out=None,
                      ws=None, stream=None):
    N, D = x.shape
    E, Dff, _ = w1.shape
    _need(x, torch.bfloat16, (N, D), "x")
    _need(w_gate, torch.bfloat16, (E, D), "w_gate")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    _need(w1, torch.bfloat16, (E, Dff, D), "w1")
    if act == ACT_SWIGLU:
        _need(w3, torch.bfloat16, (E, Dff, D), "w3")
    _need(w2, torch.bfloat16, (E, D, Dff), "w2")
    dev = x.device
    out = torch.empty((N, D), dtype=torch.bfloat16, device=dev) if out is None else out
    _need(out, torch.bfloat16, (N, D), "out")
    ws = workspace("layer", N, D, E, K, Dff, device=dev) if ws is None else ws
    _check("moe_layer_forward", load().moe_layer_forward(
        _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(w1), _ptr(w3) if act == ACT_SWIGLU else None,
        _ptr(w2), N, D, E, K, Dff, mode, act, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def moe_routing_stats(expert_offsets, ema, bias=None, decay: float = 0.99, bias_step: float = 0.1,
                      kl_out=None, stream=None):
    """EMA of per-expert fractions, KL to uniform and the bias step (in place
    on ema / bias).  Returns kl_out (a 1-element fp32 tensor)."""
    E = expert_offsets.shape[0] - 1
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _need(ema, torch.float32, (E,), "ema")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    kl_out = torch.empty(1, dtype=torch.float32, device=ema.device) if kl_out is None else kl_out
    _check("moe_routing_stats", load().moe_routing_stats(
        _ptr(expert_offsets), E, decay, bias_step, _ptr(ema), _ptr(bias), _ptr(kl_out), _stream(stream)))
    return kl_out


def layer_intermediates(ws: torch.Tensor, N, D, E, K, Dff) -> dict:
    """Views of the intermediates moe_layer_forward left in its workspace."""
    o = layer_workspace_layout(N, D, E, K, Dff)
    A = N * K

    def view(off, n, dtype, shape):
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype).view(shape)

    return dict(topk_ids=view(o[0], A, torch.int32, (N, K)),
                topk_w=view(o[1], A, torch.float32, (N, K)),
                expert_offsets=view(o[2], E + 1, torch.int32, (E + 1,)),
                perm_src=view(o[3], A, torch.int32, (A,)),
                inv_perm=view(o[4], A, torch.int32, (N, K)),
                x_perm=view(o[5], A * D, torch.bfloat16, (A, D)),
                h=view(o[6], A * Dff, torch.bfloat16, (A, Dff)),
                y_perm=view(o[7], A * D, torch.bfloat16, (A, D)))


# ---------------------------------------------------------------- paradigm B (fixed capacity)
def capacity(N: int, E: int, K: int, capacity_factor: float = 1.5) -> int:
    c = int(load().moe_capacity(N, E, K, capacity_factor))
    if c < 0:
        raise ValueError("invalid capacity arguments")
    return c


def workspace_padded(op: str, N=0, D=0, E=0, K=0, Dff=0, cap=0, device=None) -> torch.Tensor:
    n = int(load().moe_workspace_size_padded(op.encode(), N, D, E, K, Dff, cap))
    if n == 0:
        raise ValueError(f"invalid padded workspace request {op}")
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def moe_permute_padded(x, topk_ids, E: int, cap: int, expert_offsets=None, kept=None, slot=None,
                       x_pad=None, ws=None, stream=None):
    N, D = x.shape
    K = topk_ids.shape[1]
    _need(x, torch.bfloat16, (N, D), "x")
    _need(topk_ids, torch.int32, (N, K), "topk_ids")
    dev = x.device
    expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if expert_offsets is None else expert_offsets
    kept = torch.empty(E, dtype=torch.int32, device=dev) if kept is None else kept
    slot = torch.empty((N, K), dtype=torch.int32, device=dev) if slot is None else slot
    x_pad = torch.empty((E * cap, D), dtype=torch.bfloat16, device=dev) if x_pad is None else x_pad
    ws = workspace_padded("permute", N=N, E=E, cap=cap, device=dev) if ws is None else ws
    _check("moe_permute_padded", load().moe_permute_padded(
        _ptr(x), _ptr(topk_ids), N, D, E, K, cap, _ptr(expert_offsets), _ptr(kept), _ptr(slot),
        _ptr(x_pad) if x_pad.numel() else None, _ptr(ws), ws.numel(), _stream(stream)))
    return expert_offsets, kept, slot, x_pad


def moe_combine_padded(y_pad, slot, topk_w, E: int, cap: int, out=None, ws=None, stream=None):
    N, K = slot.shape
    D = y_pad.shape[1]
    _need(slot, torch.int32, (N, K), "slot")
    _need(topk_w, torch.float32, (N, K), "topk_w")
    out = torch.empty((N, D), dtype=torch.bfloat16, device=slot.device) if out is None else out
    ws = workspace("combine", device=slot.device) if ws is None else ws
    _check("moe_combine_padded", load().moe_combine_padded(
        _ptr(y_pad) if y_pad.numel() else None, _ptr(slot), _ptr(topk_w), N, D, K, E, cap, _ptr(out),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def moe_layer_forward_padded(x, w_gate, bias, w1, w3, w2, K: int, mode: int, act: int, cap: int,
                             out=None, ws=None, stream=None):
    N, D = x.shape
    E, Dff, _ = w1.shape
    _need(x, torch.bfloat16, (N, D), "x")
    dev = x.device
    out = torch.empty((N, D), dtype=torch.bfloat16, device=dev) if out is None else out
    ws = workspace_padded("layer", N, D, E, K, Dff, cap, device=dev) if ws is None else ws
    _check("moe_layer_forward_padded", load().moe_layer_forward_padded(
        _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(w1), _ptr(w3) if act == ACT_SWIGLU else None, _ptr(w2),
        N, D, E, K, Dff, mode, act, cap, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def layer_padded_intermediates(ws: torch.Tensor, N, D, E, K, Dff, cap) -> dict:
    arr = (ctypes.c_size_t * 8)()
    if load().moe_layer_padded_workspace_layout(N, D, E, K, Dff, cap, arr) != 0:
        raise ValueError("invalid sizes")
    o = list(arr)
    A, R = N * K, E * cap

    def view(off, n, dtype, shape):
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype).view(shape)

    return dict(topk_ids=view(o[0], A, torch.int32, (N, K)), topk_w=view(o[1], A, torch.float32, (N, K)),
                expert_offsets=view(o[2], E + 1, torch.int32, (E + 1,)), kept=view(o[3], E, torch.int32, (E,)),
                slot=view(o[4], A, torch.int32, (N, K)), x_pad=view(o[5], R * D, torch.bfloat16, (R, D)),
                h=view(o[6], R * Dff, torch.bfloat16, (R, Dff)), y_pad=view(o[7], R * D, torch.bfloat16, (R, D)))


# ---------------------------------------------------------------- FP8 (e4m3) experts
def moe_quantize_e4m3(src, q=None, scale=None, stream=None):
    """Per-row e4m3 quantisation of a bf16 tensor (last dim = row): returns
    (codes uint8 of src's shape, scale fp32 of src.shape[:-1])."""
    if src.dtype != torch.bfloat16 or not src.is_cuda or not src.is_contiguous():
        raise TypeError("src: expected a contiguous bf16 CUDA tensor")
    cols = src.shape[-1]
    rows = src.numel() // cols if cols else 0
    q = torch.empty(src.shape, dtype=torch.uint8, device=src.device) if q is None else q
    scale = torch.empty(src.shape[:-1], dtype=torch.float32, device=src.device) if scale is None else scale
    _need(q, torch.uint8, src.shape, "q")
    _need(scale, torch.float32, src.shape[:-1], "scale")
    _check("moe_quantize_e4m3", load().moe_quantize_e4m3(
        _ptr(src), rows, cols, _ptr(q), _ptr(scale), _stream(stream)))
    return q, scale


def quantize_experts_e4m3(w1, w3, w2, stream=None) -> dict:
    """e4m3 codes and per-output-channel scales of the three expert tensors."""
    w1q, s1 = moe_quantize_e4m3(w1, stream=stream)
    w3q, s3 = moe_quantize_e4m3(w3, stream=stream) if w3 is not None else (None, None)
    w2q, s2 = moe_quantize_e4m3(w2, stream=stream)
    return dict(w1q=w1q, s1=s1, w3q=w3q, s3=s3, w2q=w2q, s2=s2)


def moe_permute_e4m3(xq, topk_ids, E: int, expert_offsets=None, perm_src=None, inv_perm=None,
                     xq_perm=None, ws=None, stream=None):
    N, D = xq.shape
    K = topk_ids.shape[1]
    _need(xq, torch.uint8, (N, D), "xq")
    _need(topk_ids, torch.int32, (N, K), "topk_ids")
    dev = xq.device
    expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev) if expert_offsets is None else expert_offsets
    perm_src = torch.empty(N * K, dtype=torch.int32, device=dev) if perm_src is None else perm_src
    inv_perm = torch.empty((N, K), dtype=torch.int32, device=dev) if inv_perm is None else inv_perm
    xq_perm = torch.empty((N * K, D), dtype=torch.uint8, device=dev) if xq_perm is None else xq_perm
    _need(xq_perm, torch.uint8, (N * K, D), "xq_perm")
    ws = workspace("permute", N=N, E=E, device=dev) if ws is None else ws
    _check("moe_permute_e4m3", load().moe_permute_e4m3(
        _ptr(xq), _ptr(topk_ids), N, D, E, K, _ptr(expert_offsets), _ptr(perm_src),
        _ptr(inv_perm), _ptr(xq_perm), _ptr(ws), ws.numel(), _stream(stream)))
    return expert_offsets, perm_src, inv_perm, xq_perm


def moe_grouped_ffn_e4m3(xq_perm, x_scale, x_scale_index, expert_offsets, w1q, s1, w3q, s3, w2q, s2,
                         act: int, h=None, hq=None, h_scale=None, y_perm=None, ws=None, stream=None):
    rows, D = xq_perm.shape
    E, Dff, _ = w1q.shape
    _need(xq_perm, torch.uint8, (rows, D), "xq_perm")
    _need(expert_offsets, torch.int32, (E + 1,), "expert_offsets")
    _need(w1q, torch.uint8, (E, Dff, D), "w1q")
    _need(s1, torch.float32, (E, Dff), "s1")
    if act == ACT_SWIGLU:
        _need(w3q, torch.uint8, (E, Dff, D), "w3q")
        _need(s3, torch.float32, (E, Dff), "s3")
    _need(w2q, torch.uint8, (E, D, Dff), "w2q")
    _need(s2, torch.float32, (E, D), "s2")
    dev = xq_perm.device
    h = torch.empty((rows, Dff), dtype=torch.bfloat16, device=dev) if h is None else h
    hq = torch.empty((rows, Dff), dtype=torch.uint8, device=dev) if hq is None else hq
    h_scale = torch.empty(rows, dtype=torch.float32, device=dev) if h_scale is None else h_scale
    y_perm = torch.empty((rows, D), dtype=torch.bfloat16, device=dev) if y_perm is None else y_perm
    _need(h, torch.bfloat16, (rows, Dff), "h")
    _need(hq, torch.uint8, (rows, Dff), "hq")
    _need(h_scale, torch.float32, (rows,), "h_scale")
    _need(y_perm, torch.bfloat16, (rows, D), "y_perm")
    ws = workspace("ffn", rows, D, E, 1, Dff, device=dev) if ws is None else ws
    sw = act == ACT_SWIGLU
    _check("moe_grouped_ffn_e4m3", load().moe_grouped_ffn_e4m3(
        _ptr(xq_perm), _ptr(x_scale), _ptr(x_scale_index), _ptr(expert_offsets), rows, _ptr(w1q), _ptr(s1),
        _ptr(w3q) if sw else None, _ptr(s3) if sw else None, _ptr(w2q), _ptr(s2), E, D, Dff, act,
        _ptr(h), _ptr(hq), _ptr(h_scale), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))
    return h, hq, h_scale, y_perm


def moe_layer_forward_e4m3(x, w_gate, bias, qw: dict, K: int, mode: int, act: int, out=None, ws=None,
                           stream=None):
    """The layer with e4m3 experts; ``qw`` as returned by quantize_experts_e4m3."""
    N, D = x.shape
    E, Dff, _ = qw["w1q"].shape
    _need(x, torch.bfloat16, (N, D), "x")
    _need(w_gate, torch.bfloat16, (E, D), "w_gate")
    if bias is not None:
        _need(bias, torch.float32, (E,), "bias")
    dev = x.device
    out = torch.empty((N, D), dtype=torch.bfloat16, device=dev) if out is None else out
    _need(out, torch.bfloat16, (N, D), "out")
    ws = workspace("layer_e4m3", N, D, E, K, Dff, device=dev) if ws is None else ws
    sw = act == ACT_SWIGLU
    _check("moe_layer_forward_e4m3", load().moe_layer_forward_e4m3(
        _ptr(x), _ptr(w_gate), _ptr(bias), _ptr(qw["w1q"]), _ptr(qw["s1"]),
        _ptr(qw["w3q"]) if sw else None, _ptr(qw["s3"]) if sw else None, _ptr(qw["w2q"]), _ptr(qw["s2"]),
        N, D, E, K, Dff, mode, act, _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def layer_launches_e4m3(N, D, E, K, Dff, act) -> int:
    return int(load().moe_layer_launches_e4m3(N, D, E, K, Dff, act))


def layer_e4m3_intermediates(ws: torch.Tensor, N, D, E, K, Dff) -> dict:
    """Views of the intermediates moe_layer_forward_e4m3 left in its workspace."""
    arr = (ctypes.c_size_t * 12)()
    if load().moe_layer_e4m3_workspace_layout(N, D, E, K, Dff, arr) != 0:
        raise ValueError("invalid sizes")
    o = list(arr)
    A = N * K

    def view(off, n, dtype, shape):
        nbytes = n * torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + nbytes].view(dtype).view(shape)

    return dict(topk_ids=view(o[0], A, torch.int32, (N, K)), topk_w=view(o[1], A, torch.float32, (N, K)),
                expert_offsets=view(o[2], E + 1, torch.int32, (E + 1,)), perm_src=view(o[3], A, torch.int32, (A,)),
                inv_perm=view(o[4], A, torch.int32, (N, K)), xq=view(o[5], N * D, torch.uint8, (N, D)),
                x_scale=view(o[6], N, torch.float32, (N,)), xq_perm=view(o[7], A * D, torch.uint8, (A, D)),
                h=view(o[8], A * Dff, torch.bfloat16, (A, Dff)), hq=view(o[9], A * Dff, torch.uint8, (A, Dff)),
                h_scale=view(o[10], A, torch.float32, (A,)), y_perm=view(o[11], A * D, torch.bfloat16, (A, D)))


def moe_grouped_ffn_e4m3_gathered(xq, x_scale, perm_src, expert_offsets, w1q, s1, w3q, s3, w2q, s2, act: int,
                                  h=None, hq=None, h_scale=None, y_perm=None, ws=None, stream=None):
    """moe_grouped_ffn_e4m3 with GEMM1 reading token codes of xq through perm_src."""
    N, D = xq.shape
    rows = perm_src.shape[0]
    E, Dff, _ = w1q.shape
    _need(xq, torch.uint8, (N, D), "xq")
    _need(x_scale, torch.float32, (N,), "x_scale")
    _need(perm_src, torch.int32, (rows,), "perm_src")
    dev = xq.device
    h = torch.empty((rows, Dff), dtype=torch.bfloat16, device=dev) if h is None else h
    hq = torch.empty((rows, Dff), dtype=torch.uint8, device=dev) if hq is None else hq
    h_scale = torch.empty(rows, dtype=torch.float32, device=dev) if h_scale is None else h_scale
    y_perm = torch.empty((rows, D), dtype=torch.bfloat16, device=dev) if y_perm is None else y_perm
    ws = workspace("ffn", rows, D, E, 1, Dff, device=dev) if ws is None else ws
    sw = act == ACT_SWIGLU
    _check("moe_grouped_ffn_e4m3_gathered", load().moe_grouped_ffn_e4m3_gathered(
        _ptr(xq), _ptr(x_scale), N, _ptr(perm_src), _ptr(expert_offsets), rows, _ptr(w1q), _ptr(s1),
        _ptr(w3q) if sw else None, _ptr(s3) if sw else None, _ptr(w2q), _ptr(s2), E, D, Dff, act,
        _ptr(h), _ptr(hq), _ptr(h_scale), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)))
    return h, hq, h_scale, y_perm
