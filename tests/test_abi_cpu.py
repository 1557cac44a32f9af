"""CPU checks of the C-ABI library: it builds, loads, exports every entry point
include/moe.h declares, and its host-side validation rejects bad arguments
before anything reaches the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_layer_02_gb300 import build, moe
    build.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", text, re.M)))


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_layer_forward"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from mixture_experts_layer_02_gb300 import moe
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in moe.h but not exported"
    assert set(declared_functions()) == set(moe.EXPORTED)


def test_status_strings_and_version(lib):
    assert lib.moe_status_string(0) == b"ok"
    assert b"timed out" in lib.moe_status_string(6)
    assert b"sm_103a" in lib.moe_version()


def test_workspace_sizes(lib):
    from mixture_experts_layer_02_gb300 import moe
    assert moe.workspace_size("combine") == 256
    # route: header + fp32 partials [splits][N][E rounded up to 32]
    assert moe.workspace_size("route", 4096, 7168, 256, 8) >= 256 + 4096 * 256 * 4
    assert moe.workspace_size("route", 1, 2048, 128, 8) >= 256 + 128 * 4
    assert moe.workspace_size("route", 4, 100, 8, 2) == 0
    # ffn: header only when the call fills the GPU, partials for decode sizes
    assert moe.workspace_size("ffn", 8192, 4096, 8, 1, 14336) == 256
    assert moe.workspace_size("ffn", 8, 2048, 128, 1, 768) > 256
    # permute: header + [E][ceil(N/16)] + [E] ints, 256-aligned
    n = moe.workspace_size("permute", N=4096, E=256)
    assert n >= 256 + (256 * 256 + 256) * 4
    lay = moe.layer_workspace_layout(64, 128, 8, 2, 256)
    assert lay == sorted(lay) and all(o % 256 == 0 for o in lay)
    total = moe.workspace_size("layer", 64, 128, 8, 2, 256)
    assert total >= lay[-1] + 128 * 128 * 2
    assert moe.workspace_size("layer", 64, 100, 8, 2, 256) == 0       # D not a multiple of 64
    assert moe.workspace_size("bogus", 1, 64, 1, 1, 64) == 0


def _call_route(lib, N=4, D=64, E=8, K=2, mode=0, ws=1024, ws_bytes=4096):
    p = ctypes.c_void_p
    return lib.moe_route(p(4096), p(8192), None, N, D, E, K, mode, p(12288), p(16384), None,
                         p(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=0), 1), (dict(K=9), 1), (dict(E=0), 1), (dict(E=2048, K=2), 1), (dict(K=33, E=64), 1),
    (dict(D=100), 1), (dict(N=-1), 1), (dict(mode=5), 1), (dict(ws=0), 1),
    (dict(ws=1032), 1),                     # misaligned workspace
    (dict(ws_bytes=8), 3),                  # workspace too small
])
def test_route_validation(lib, kw, status):
    assert _call_route(lib, **kw) == status
    assert lib.moe_last_error_detail() != b""


def test_other_entry_points_validate(lib):
    p = ctypes.c_void_p
    # permute: NULL x with N > 0
    assert lib.moe_permute(None, p(4096), 4, 64, 8, 2, p(256), p(512), p(768), p(1024), p(2048),
                           1 << 20, None) == 1
    # grouped FFN: SwiGLU without w3
    assert lib.moe_grouped_ffn(p(4096), p(256), 8, p(8192), None, p(12288), 8, 64, 128, 1,
                               p(16384), p(20480), p(2048), 1 << 20, None) == 1
    # grouped FFN: Dff not a multiple of 64
    assert lib.moe_grouped_ffn(p(4096), p(256), 8, p(8192), p(8192), p(12288), 8, 64, 100, 1,
                               p(16384), p(20480), p(2048), 1 << 20, None) == 1
    # combine: misaligned out
    assert lib.moe_combine(p(4096), p(256), p(512), 4, 64, 2, p(1000), p(2048), 256, None) == 1
    # layer: workspace too small
    assert lib.moe_layer_forward(p(4096), p(4096), None, p(4096), p(4096), p(4096), 64, 128, 8, 2,
                                 256, 0, 1, p(8192), p(2048), 1024, None) == 3
    # layer: bad activation
    assert lib.moe_layer_forward(p(4096), p(4096), None, p(4096), p(4096), p(4096), 64, 128, 8, 2,
                                 256, 0, 7, p(8192), p(2048), 1 << 30, None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    from mixture_experts_layer_02_gb300 import moe
    import importlib
    m = importlib.reload(moe)
    with pytest.raises(RuntimeError, match="libmoe.so not found"):
        m._lib = None
        m.load(str(tmp_path / "missing.so"))
    importlib.reload(moe)
