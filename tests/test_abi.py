"""Host-side checks of the C ABI (no GPU needed).

The library builds for sm_103a, loads, exports every function the header
declares with the Python binding's signature, and rejects bad arguments on the
host before any CUDA call (these calls return before touching a device).
"""
import ctypes
import os
import re

import pytest

from moe_routing_precision_gb300 import _build

HEADER = os.path.join(_build.INCLUDE, "moe_route.h")


@pytest.fixture(scope="session")
def L():
    _build.build()
    from moe_routing_precision_gb300 import ops
    return ops.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keywords = {"if", "sizeof", "defined"}
    return sorted(set(n for n in names if n not in keywords))


def test_header_declares_the_five_ops():
    names = _declared_functions()
    for op in ("moe_topk_gate", "moe_route_map", "moe_expand_cast_fp8", "swiglu_cast_fp8",
               "moe_combine"):
        assert op in names


def test_library_exports_every_declared_symbol(L):
    from moe_routing_precision_gb300 import ops
    names = _declared_functions()
    assert set(names) == set(ops.SIGNATURES), set(names) ^ set(ops.SIGNATURES)
    for n in names:
        assert hasattr(L, n), n


def test_abi_version_and_status_strings(L):
    assert L.moe_abi_version() == 1
    for rc in range(5):
        assert L.moe_status_string(rc)
    assert b"unknown" in L.moe_status_string(99)


def test_workspace_size(L):
    assert L.moe_route_map_workspace_bytes(0, 256, 8) == 0
    assert L.moe_route_map_workspace_bytes(1, 256, 8) == 1024
    # about 128 chunks of a multiple of 32 tokens: 512 tokens per chunk at T=65536
    assert L.moe_route_map_workspace_bytes(65536, 256, 8) == 128 * 256 * 4
    # chunks stop growing at 512 tokens: T=2^21 -> 4096 chunks
    assert L.moe_route_map_workspace_bytes(1 << 21, 256, 8) == 4096 * 256 * 4
    # small T: 32-token chunks
    assert L.moe_route_map_workspace_bytes(100, 16, 2) == 256
    assert L.moe_route_map_workspace_bytes(129, 16, 2) % 256 == 0
    assert L.moe_route_map_workspace_bytes(100, 16, 0) == 0


FAKE = 0x10000  # never dereferenced: every call below is rejected on the host
INVALID, UNSUPPORTED = 1, 2


def test_topk_gate_rejects_bad_arguments(L):
    f = L.moe_topk_gate
    assert f(FAKE, 4, 0, 1, FAKE, FAKE, 1, None) == INVALID          # E = 0
    assert f(FAKE, 4, 1025, 1, FAKE, FAKE, 1, None) == INVALID       # E > max
    assert f(FAKE, 4, 16, 17, FAKE, FAKE, 1, None) == INVALID        # k > E
    assert f(FAKE, 4, 64, 33, FAKE, FAKE, 1, None) == INVALID        # k > 32
    assert f(FAKE, 4, 16, 0, FAKE, FAKE, 1, None) == INVALID         # k = 0
    assert f(FAKE, -1, 16, 2, FAKE, FAKE, 1, None) == INVALID        # T < 0
    assert f(None, 4, 16, 2, FAKE, FAKE, 1, None) == INVALID         # null scores
    assert f(FAKE, 4, 16, 2, FAKE, None, 1, None) == INVALID         # null weights
    assert f(FAKE + 2, 4, 16, 2, FAKE, FAKE, 1, None) == INVALID     # misaligned
    assert f(FAKE, 4, 16, 2, FAKE, FAKE, 7, None) == INVALID         # bad mode
    assert f(None, 0, 16, 2, None, None, 1, None) == 0               # T = 0: no-op


def test_route_map_rejects_bad_arguments(L):
    f = L.moe_route_map
    ws = L.moe_route_map_workspace_bytes(100, 16, 2)
    assert f(FAKE, 100, 16, 2, FAKE, FAKE, FAKE, FAKE, FAKE, ws - 1, None) == INVALID
    assert f(FAKE, 100, 16, 2, FAKE, FAKE, FAKE, FAKE, None, ws, None) == INVALID
    assert f(FAKE, 100, 16, 2, FAKE, FAKE, FAKE, FAKE, FAKE + 4, ws, None) == INVALID
    assert f(FAKE, 100, 16, 17, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None) == INVALID
    assert f(FAKE, 1 << 27, 16, 16, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == INVALID


def test_expand_cast_rejects_bad_arguments(L):
    f = L.moe_expand_cast_fp8
    assert f(FAKE, 4, 256, 2, FAKE, 8, FAKE, FAKE, 64, None) == UNSUPPORTED   # group
    assert f(FAKE, 4, 200, 2, FAKE, 8, FAKE, FAKE, 128, None) == INVALID      # H % 128
    assert f(FAKE + 8, 4, 256, 2, FAKE, 8, FAKE, FAKE, 128, None) == INVALID  # x align
    assert f(FAKE, 4, 256, 2, FAKE, 8, FAKE + 4, FAKE, 128, None) == INVALID  # out align
    assert f(FAKE, 4, 256, 0, FAKE, 8, FAKE, FAKE, 128, None) == INVALID      # k = 0
    assert f(FAKE, 4, 256, 2, None, 8, FAKE, FAKE, 128, None) == INVALID      # null pos
    assert f(None, 0, 256, 2, None, 0, None, None, 128, None) == 0            # T = 0


def test_swiglu_rejects_bad_arguments(L):
    f = L.swiglu_cast_fp8
    assert f(FAKE, 4, 2048, FAKE, FAKE, 32, None) == UNSUPPORTED
    assert f(FAKE, 4, 100, FAKE, FAKE, 128, None) == INVALID
    assert f(FAKE, 4, 2048, None, FAKE, 128, None) == INVALID
    assert f(FAKE + 2, 4, 2048, FAKE, FAKE, 128, None) == INVALID
    assert f(None, 0, 2048, None, None, 128, None) == 0


def test_combine_rejects_bad_arguments(L):
    f = L.moe_combine
    assert f(FAKE, FAKE, FAKE, 4, 12, 2, 8, FAKE, 0, None) == INVALID      # H % 8
    assert f(FAKE, FAKE, FAKE, 4, 256, 2, 8, FAKE, 5, None) == INVALID     # dtype
    assert f(FAKE, FAKE, FAKE, 4, 256, 2, 8, FAKE + 8, 0, None) == INVALID  # out align
    assert f(FAKE, None, FAKE, 4, 256, 2, 8, FAKE, 0, None) == INVALID
    assert f(None, None, None, 0, 256, 2, 0, None, 0, None) == 0


def test_peak_copy_rejects_bad_arguments(L):
    assert L.moe_peak_copy(FAKE, FAKE, 17, None) == INVALID
    assert L.moe_peak_copy(FAKE + 1, FAKE, 32, None) == INVALID
    assert L.moe_peak_copy(None, None, 0, None) == 0


def test_no_kernel_launched_by_rejected_calls(L):
    assert L.moe_kernel_launch_count() == 0


def test_binding_refuses_cpu_tensors():
    import torch
    from moe_routing_precision_gb300 import ops
    _build.build()
    with pytest.raises(ValueError, match="CUDA"):
        ops.topk_gate(torch.zeros(4, 16), 2)
    with pytest.raises(ValueError, match="CUDA"):
        ops.swiglu_cast_fp8(torch.zeros(4, 256, dtype=torch.bfloat16))


def test_padded_entry_points_reject_bad_arguments(L):
    f = L.moe_route_map_aligned
    ws = L.moe_route_map_workspace_bytes(100, 16, 2)
    args = lambda align, rows: (FAKE, 100, 16, 2, align, rows, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None)
    assert f(*args(0, 1000)) == INVALID                  # align 0
    assert f(*args(8192, 1000)) == INVALID               # align > 4096
    assert f(*args(4, -1)) == INVALID                    # negative rows
    assert f(*args(4, 1 << 31)) == INVALID               # rows >= 2^31
    assert f(FAKE, 100, 16, 2, 4, 1000, FAKE, FAKE, FAKE, None, FAKE, ws, None) == INVALID
    g = L.moe_expand_cast_fp8_padded
    assert g(FAKE, 4, 256, 2, FAKE, FAKE, 20, FAKE, FAKE, 64, None) == UNSUPPORTED
    assert g(FAKE, 4, 256, 2, FAKE, None, 20, FAKE, FAKE, 128, None) == INVALID   # no sorted_src
    assert g(FAKE, 4, 256, 2, FAKE, FAKE + 2, 20, FAKE, FAKE, 128, None) == INVALID
    assert g(None, 0, 256, 2, None, None, 0, None, None, 128, None) == 0          # nothing to do


def test_cast_option_entry_points_reject_bad_arguments(L):
    f = L.moe_expand_cast_fp8_ex
    args = lambda flags, ld, sf=FAKE, R=20, ws=None, wsb=0: (
        FAKE, 4, 512, 2, FAKE, FAKE, R, FAKE, sf, flags, ld, ws, wsb, 128, None)
    assert f(*args(4, 0)) == INVALID                     # UE8M0 without POW2
    assert f(*args(8, 0)) == INVALID                     # unknown flag
    assert f(*args(1, 18)) == INVALID                    # ld < rows
    assert f(*args(1, 22)) == INVALID                    # ld not a multiple of 4
    assert f(*args(3, 1 << 31)) == INVALID               # ld >= 2^31
    assert f(*args(2, 0, sf=FAKE + 2)) == INVALID        # f32 scales 4-byte aligned
    assert f(*args(7, 20, sf=FAKE + 2)) == INVALID       # packed words 4-byte aligned
    need = L.moe_expand_cast_fp8_ex_workspace_bytes(4, 512, 7)
    assert need == 256                                   # 4 tokens x 1 word, rounded to 256
    assert L.moe_expand_cast_fp8_ex_workspace_bytes(4, 512, 3) == 256
    assert L.moe_expand_cast_fp8_ex_workspace_bytes(1000, 7168, 1) == (1000 * 56 * 4 + 255) // 256 * 256
    assert L.moe_expand_cast_fp8_ex_workspace_bytes(1000, 7168, 7) == (1000 * 56 + 255) // 256 * 256
    assert L.moe_expand_cast_fp8_ex_workspace_bytes(1000, 7168, 6) == 0   # row-major: none
    assert f(*args(7, 20, ws=FAKE, wsb=need - 1)) == INVALID        # workspace too small
    assert f(*args(7, 20, ws=FAKE + 8, wsb=need)) == INVALID        # workspace 16-byte aligned
    assert f(FAKE, 4, 512, 2, FAKE, None, 20, FAKE, FAKE, 0, 0, None, 0, 64, None) == UNSUPPORTED
    assert f(None, 0, 512, 2, None, None, 0, None, None, 7, 0, None, 0, 128, None) == 0
    g = L.swiglu_cast_fp8_ex
    sargs = lambda flags=0, ld=0, has_clamp=0, clamp=0.0, w=None, cnt=None: (
        FAKE, 4, 512, FAKE, FAKE, flags, ld, has_clamp, clamp, w, cnt, 128, None)
    assert g(*sargs(flags=4)) == INVALID
    assert g(*sargs(flags=1, ld=2)) == INVALID
    assert g(*sargs(has_clamp=1, clamp=-1.0)) == INVALID
    assert g(*sargs(has_clamp=1, clamp=float("nan"))) == INVALID
    assert g(*sargs(has_clamp=1, clamp=float("inf"))) == INVALID
    assert g(*sargs(w=FAKE + 2)) == INVALID              # weights 4-byte aligned
    assert g(*sargs(cnt=FAKE + 4)) == INVALID            # counter 8-byte aligned
    assert g(None, 0, 512, None, None, 7, 0, 1, 1.0, None, None, 128, None) == 0
    assert L.moe_kernel_launch_count() == 0


def test_route_expand_cast_rejects_bad_arguments(L):
    f = L.moe_route_expand_cast_fp8
    T, E, k, H = 8, 256, 8, 512
    need = L.moe_route_expand_cast_fp8_workspace_bytes(T, E, k)
    assert need >= 256 + L.moe_route_map_workspace_bytes(T, E, k)
    # the chained path's histogram: one row of E counters per chunk of 16 to 64 tokens
    for TT, chunk in ((8, 16), (16385, 32), (65536, 64)):
        rows = -(-TT // chunk)
        assert L.moe_route_expand_cast_fp8_workspace_bytes(TT, E, k) >= 256 + rows * E * 4
    def args(mode=0, H=H, x=FAKE, ws=FAKE, wsb=need, group=128):
        return (FAKE, T, E, k, x, H, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, wsb,
                mode, group, None)
    assert f(*args(mode=5)) == INVALID
    assert f(*args(mode=-1)) == INVALID
    assert f(*args(mode=3, wsb=need - 1)) == INVALID   # REPLICATED checks the same arguments
    assert f(*args(group=64)) == UNSUPPORTED
    assert f(*args(H=200)) == INVALID
    assert f(*args(wsb=need - 1)) == INVALID
    assert f(*args(ws=FAKE + 8)) == INVALID         # workspace 16-byte aligned
    assert f(*args(x=FAKE + 4)) == INVALID          # x 16-byte aligned
    assert f(*args(ws=None)) == INVALID
    assert L.moe_debug_set(99, 0) == INVALID
    assert L.moe_debug_set(1, 10) == INVALID        # timeout below 1 us
    assert L.moe_debug_set(1, 61 * 10**9) == INVALID
    assert L.moe_debug_set(1, 10**9) == 0
    assert L.moe_debug_set(2, 0) == 0
    assert L.moe_kernel_launch_count() == 0


def test_fp4_entry_point_rejects_bad_arguments(L):
    f = L.moe_expand_cast_fp4
    def args(H=512, group=32, flags=0, ld=0, x=FAKE, out=FAKE, ws=None, wsb=0):
        return (x, 4, H, 2, FAKE, FAKE, 8, out, FAKE, flags, ld, ws, wsb, group, None)
    assert f(*args(group=48)) == UNSUPPORTED
    assert f(*args(group=256)) == UNSUPPORTED
    assert f(*args(H=496)) == INVALID               # H % 32
    assert f(*args(H=384, group=256)) == UNSUPPORTED
    assert f(*args(H=288, group=128)) == INVALID     # H % group
    assert f(*args(H=32768)) == UNSUPPORTED
    assert f(*args(flags=4)) == INVALID              # UE8M0 without POW2
    assert f(*args(flags=1, ld=6)) == INVALID        # ld < rows
    assert f(*args(x=FAKE + 8)) == INVALID
    assert f(*args(out=FAKE + 8)) == INVALID
    need = L.moe_expand_cast_fp4_workspace_bytes(4, 512, 32, 1)
    assert need == 256 and L.moe_expand_cast_fp4_workspace_bytes(4, 512, 32, 2) == 0
    assert L.moe_expand_cast_fp4_workspace_bytes(1000, 7168, 32, 1) == (1000 * 224 * 4 + 255) // 256 * 256
    assert f(*args(flags=1, ld=8, ws=FAKE, wsb=need - 1)) == INVALID
    assert L.moe_kernel_launch_count() == 0


def test_swiglu_fp4_rejects_bad_arguments(L):
    f = L.swiglu_cast_fp4
    args = lambda n=512, group=32, flags=0, ld=0, x=FAKE: (x, 4, n, FAKE, FAKE, flags, ld, 0, 0.0,
                                                          None, None, group, None)
    assert f(*args(group=8)) == UNSUPPORTED
    assert f(*args(n=496)) == INVALID
    assert f(*args(n=288, group=128)) == INVALID
    assert f(*args(flags=4)) == INVALID
    assert f(*args(x=FAKE + 8)) == INVALID
    assert f(None, 0, 512, None, None, 0, 0, 0, 0.0, None, None, 32, None) == 0
    assert L.moe_kernel_launch_count() == 0


def test_debug_cvt_rejects_bad_arguments(L):
    f = L.moe_debug_cvt
    assert f(2, FAKE, FAKE, 16, None) == INVALID          # unknown format
    assert f(0, FAKE, FAKE, 6, None) == INVALID           # n % 4
    assert f(1, FAKE + 4, FAKE, 16, None) == INVALID      # alignment
    assert f(0, None, None, 0, None) == 0
    assert L.moe_kernel_launch_count() == 0


def test_debug_bounds_entry_points_of_the_normal_library(L):
    """The normal library reports no debug checks and refuses the self-test
    without launching anything."""
    from moe_routing_precision_gb300 import ops
    n = L.moe_kernel_launch_count()
    assert L.moe_debug_bounds_enabled() == 0
    assert L.moe_debug_bounds_selftest(None) == ops.MOE_ERR_UNSUPPORTED
    assert L.moe_kernel_launch_count() == n


def test_debug_bounds_library_builds_and_exports_every_symbol():
    """libmoe_route_debug.so (the sources with MOE_DEBUG_BOUNDS defined)
    builds, exports the header's symbols, says it is the debug build, and
    rejects bad arguments on the host exactly as the normal library does."""
    from moe_routing_precision_gb300 import ops
    path = _build.build(debug_bounds=True)
    assert path == _build.DEBUG_LIB_PATH and path != _build.LIB_PATH
    D = ops.load_library(path)
    for n in _declared_functions():
        assert hasattr(D, n), n
    assert D.moe_debug_bounds_enabled() == 1
    assert D.moe_abi_version() == 1
    assert D.moe_topk_gate(FAKE, 4, 16, 17, FAKE, FAKE, 1, None) == INVALID
    assert D.moe_peak_copy(FAKE + 1, FAKE, 32, None) == INVALID
    assert D.moe_kernel_launch_count() == 0


def test_library_choice_follows_the_environment(monkeypatch):
    monkeypatch.setenv("MOE_DEBUG_BOUNDS", "1")
    assert _build.lib_path() == _build.DEBUG_LIB_PATH
    monkeypatch.setenv("MOE_DEBUG_BOUNDS", "0")
    assert _build.lib_path() == _build.LIB_PATH
    monkeypatch.delenv("MOE_DEBUG_BOUNDS")
    assert _build.lib_path() == _build.LIB_PATH
