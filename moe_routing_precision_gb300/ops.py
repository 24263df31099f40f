"""Thin Python binding of ``include/moe_route.h`` (argument marshalling only).

Every function checks dtype, device, shape and contiguity, allocates any
output the caller did not pass (PyTorch is the memory manager), and calls the
C ABI with raw device pointers and the current CUDA stream.  All computation
happens in the CUDA kernels of ``libmoe_route.so``; there is no fallback: if
the library is missing or the tensors are not on a CUDA device, the call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import lib_path

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(5)
MOE_WEIGHTS_NONE, MOE_WEIGHTS_SOFTMAX_TOPK = 0, 1
MOE_OUT_BF16, MOE_OUT_F32 = 0, 1
MOE_DEVERR_EXPERT_RANGE, MOE_DEVERR_POS_RANGE, MOE_DEVERR_DUPLICATE_EXPERT = 0x1, 0x2, 0x4
MOE_DEVERR_ROWS_SHORT, MOE_DEVERR_TIMEOUT, MOE_DEVERR_BOUNDS = 0x8, 0x10, 0x20
GROUP = 128
SF_COLMAJOR, SF_POW2, SF_UE8M0 = 0x1, 0x2, 0x4

# Every symbol declared in include/moe_route.h, with its ctypes signature.
_P = ctypes.c_void_p
_i64, _i32, _sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
SIGNATURES = {
    "moe_topk_gate": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _P, _i32, _P]),
    "moe_route_map_workspace_bytes": (_sz, [_i64, _i32, _i32]),
    "moe_route_map": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _P, _P, _P, _P, _sz, _P]),
    "moe_route_map_noalloc": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _P, _P, _P, _P]),
    "moe_expand_cast_fp8": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _i64, _P, _P, _i32, _P]),
    "moe_route_map_aligned": (ctypes.c_int, [_P, _i64, _i32, _i32, _i32, _i64, _P, _P, _P, _P,
                                             _P, _sz, _P]),
    "moe_expand_cast_fp8_padded": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _P, _i64, _P, _P,
                                                  _i32, _P]),
    "swiglu_cast_fp8": (ctypes.c_int, [_P, _i64, _i32, _P, _P, _i32, _P]),
    "moe_expand_cast_fp8_ex": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _P, _i64, _P, _P,
                                              ctypes.c_uint32, _i64, _P, ctypes.c_size_t, _i32,
                                              _P]),
    "moe_expand_cast_fp8_ex_workspace_bytes": (ctypes.c_size_t, [_i64, _i32, ctypes.c_uint32]),
    "moe_expand_cast_fp4": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _P, _i64, _P, _P,
                                           ctypes.c_uint32, _i64, _P, ctypes.c_size_t, _i32, _P]),
    "moe_expand_cast_fp4_workspace_bytes": (ctypes.c_size_t, [_i64, _i32, _i32,
                                                              ctypes.c_uint32]),
    "swiglu_cast_fp4": (ctypes.c_int, [_P, _i64, _i32, _P, _P, ctypes.c_uint32, _i64, _i32,
                                       ctypes.c_float, _P, _P, _i32, _P]),
    "moe_route_expand_cast_fp8": (ctypes.c_int, [_P, _i64, _i32, _i32, _P, _i32, _P, _P, _P, _P,
                                                 _P, _P, _P, _P, _P, ctypes.c_size_t, _i32, _i32,
                                                 _P]),
    "moe_route_expand_cast_fp8_workspace_bytes": (ctypes.c_size_t, [_i64, _i32, _i32]),
    "moe_debug_set": (ctypes.c_int, [_i32, _i64]),
    "moe_debug_cvt": (ctypes.c_int, [_i32, _P, _P, _i64, _P]),
    "swiglu_cast_fp8_ex": (ctypes.c_int, [_P, _i64, _i32, _P, _P, ctypes.c_uint32, _i64, _i32,
                                          ctypes.c_float, _P, _P, _i32, _P]),
    "moe_combine": (ctypes.c_int, [_P, _P, _P, _i64, _i32, _i32, _i64, _P, _i32, _P]),
    "moe_peak_copy": (ctypes.c_int, [_P, _P, _sz, _P]),
    "moe_get_device_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_last_cuda_error_string": (ctypes.c_char_p, []),
    "moe_abi_version": (ctypes.c_int32, []),
    "moe_kernel_launch_count": (ctypes.c_uint64, []),
    "moe_debug_bounds_enabled": (ctypes.c_int32, []),
    "moe_debug_bounds_selftest": (ctypes.c_int, [_P]),
}

_lock = threading.Lock()
_lib = None


def load_library(path: str) -> ctypes.CDLL:
    """Load a build of the library at `path` and set every signature."""
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib() -> ctypes.CDLL:
    """The loaded ``libmoe_route.so``, or ``libmoe_route_debug.so`` when the
    environment variable MOE_DEBUG_BOUNDS is 1 at the first call (raises if
    it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with moe_routing_precision_gb300.build() "
                    "(nvcc, sm_103a); there is no CPU fallback")
            _lib = load_library(path)
    return _lib



class MoeError(RuntimeError):
    def __init__(self, rc: int, what: str):
        L = lib()
        msg = L.moe_status_string(rc).decode()
        if rc == MOE_ERR_CUDA:
            msg += f" ({L.moe_last_cuda_error_string().decode()})"
        super().__init__(f"{what}: {msg}")
        self.rc = rc


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _dev(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device (no CPU path), got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _ptr(t):
    return None if t is None else (t.data_ptr() or None)


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


# --------------------------------------------------------------------------

def topk_gate(scores: torch.Tensor, k: int, weights: bool = True, *, out_idx=None, out_w=None,
              stream=None):
    """Top-k experts per token (ties -> lower index) and softmax top-k weights.

    scores [T, E] float32 -> (idx [T, k] int32, w [T, k] float32 or None)."""
    _dev(scores, "scores", torch.float32)
    T, E = scores.shape
    idx = out_idx if out_idx is not None else _empty((T, k), torch.int32, scores)
    _dev(idx, "out_idx", torch.int32, (T, k))
    w = None
    if weights:
        w = out_w if out_w is not None else _empty((T, k), torch.float32, scores)
        _dev(w, "out_w", torch.float32, (T, k))
    rc = lib().moe_topk_gate(_ptr(scores), T, E, k, _ptr(idx), _ptr(w),
                             MOE_WEIGHTS_SOFTMAX_TOPK if weights else MOE_WEIGHTS_NONE,
                             _stream(stream))
    _check(rc, "moe_topk_gate")
    return idx, w


def route_map_workspace_bytes(T: int, E: int, k: int) -> int:
    return int(lib().moe_route_map_workspace_bytes(T, E, k))


def route_map(topk_idx: torch.Tensor, num_experts: int, *, workspace=None, out=None, stream=None):
    """Stable token -> expert mapping.

    topk_idx [T, k] int32 -> (counts [E], offsets [E+1], pos [T, k],
    sorted_src [T*k]), all int32.  ``workspace`` (uint8, at least
    route_map_workspace_bytes bytes) is allocated when not given."""
    _dev(topk_idx, "topk_idx", torch.int32)
    T, k = topk_idx.shape
    E = int(num_experts)
    if out is None:
        counts = _empty((E,), torch.int32, topk_idx)
        offsets = _empty((E + 1,), torch.int32, topk_idx)
        pos = _empty((T, k), torch.int32, topk_idx)
        src = _empty((T * k,), torch.int32, topk_idx)
    else:
        counts, offsets, pos, src = out
    _dev(counts, "counts", torch.int32, (E,))
    _dev(offsets, "offsets", torch.int32, (E + 1,))
    _dev(pos, "pos", torch.int32, (T, k))
    _dev(src, "sorted_src", torch.int32, (T * k,))
    need = route_map_workspace_bytes(T, E, k)
    if workspace is None:
        workspace = _empty((max(need, 1),), torch.uint8, topk_idx)
    _dev(workspace, "workspace", torch.uint8)
    rc = lib().moe_route_map(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets), _ptr(pos),
                             _ptr(src), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "moe_route_map")
    return counts, offsets, pos, src


def route_map_aligned(topk_idx: torch.Tensor, num_experts: int, align: int,
                      num_rows: int | None = None, *, workspace=None, stream=None):
    """Route map into a padded layout: each expert's segment rounded up to a
    multiple of `align` rows.  num_rows defaults to T*k + E*(align-1), which
    always suffices.  -> (counts [E], offsets [E+1] padded, pos [T, k],
    sorted_src [num_rows], -1 on padding rows), all int32."""
    _dev(topk_idx, "topk_idx", torch.int32)
    T, k = topk_idx.shape
    E = int(num_experts)
    R = T * k + E * (align - 1) if num_rows is None else int(num_rows)
    counts = _empty((E,), torch.int32, topk_idx)
    offsets = _empty((E + 1,), torch.int32, topk_idx)
    pos = _empty((T, k), torch.int32, topk_idx)
    src = _empty((R,), torch.int32, topk_idx)
    need = route_map_workspace_bytes(T, E, k)
    if workspace is None:
        workspace = _empty((max(need, 1),), torch.uint8, topk_idx)
    _dev(workspace, "workspace", torch.uint8)
    rc = lib().moe_route_map_aligned(_ptr(topk_idx), T, E, k, int(align), R, _ptr(counts),
                                     _ptr(offsets), _ptr(pos), _ptr(src), _ptr(workspace),
                                     workspace.numel(), _stream(stream))
    _check(rc, "moe_route_map_aligned")
    return counts, offsets, pos, src


def expand_cast_fp8_padded(x: torch.Tensor, pos: torch.Tensor, sorted_src: torch.Tensor, *,
                           out=None, out_sf=None, stream=None):
    """expand_cast_fp8 into a padded layout of len(sorted_src) rows, zeroing
    (codes and scales) every row whose sorted_src entry is negative."""
    _dev(x, "x", torch.bfloat16)
    _dev(pos, "pos", torch.int32)
    _dev(sorted_src, "sorted_src", torch.int32)
    T, H = x.shape
    k = pos.shape[1]
    R = sorted_src.shape[0]
    q = out if out is not None else _empty((R, H), torch.uint8, x)
    sf = out_sf if out_sf is not None else _empty((R, H // GROUP), torch.float32, x)
    _dev(q, "out", torch.uint8, (R, H))
    _dev(sf, "out_sf", torch.float32, (R, H // GROUP))
    rc = lib().moe_expand_cast_fp8_padded(_ptr(x), T, H, k, _ptr(pos), _ptr(sorted_src), R,
                                          _ptr(q), _ptr(sf), GROUP, _stream(stream))
    _check(rc, "moe_expand_cast_fp8_padded")
    return q, sf


def sf_empty(rows: int, G: int, flags: int, ld: int | None, like: torch.Tensor):
    """Scale buffer of the layout `flags` names: f32 [rows, G] or [G, ld];
    uint8 [rows, G]; or packed words as uint8 [ceil(G/4), ld, 4]."""
    ld = rows if ld is None else ld
    if flags & SF_UE8M0:
        if flags & SF_COLMAJOR:
            return _empty(((G + 3) // 4, ld, 4), torch.uint8, like), ld
        return _empty((rows, G), torch.uint8, like), ld
    if flags & SF_COLMAJOR:
        return _empty((G, ld), torch.float32, like), ld
    return _empty((rows, G), torch.float32, like), ld


PATH_AUTO, PATH_FUSED, PATH_SEPARATE, PATH_REPLICATED, PATH_CHAINED = 0, 1, 2, 3, 4
DEBUG_WAIT_TIMEOUT_NS, DEBUG_SKIP_ROUTE_SIGNAL = 1, 2


def route_expand_cast_workspace(T: int, E: int, k: int, like: torch.Tensor) -> torch.Tensor:
    """A zero-filled workspace for route_expand_cast_fp8 (its first 256 bytes
    are the fused path's control words, which must start at zero)."""
    n = int(lib().moe_route_expand_cast_fp8_workspace_bytes(T, E, k))
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=like.device)


def route_expand_cast_fp8(scores: torch.Tensor, x: torch.Tensor, k: int, *, mode: int = PATH_AUTO,
                          workspace=None, out=None, stream=None):
    """topk_gate + route_map + expand_cast_fp8 in one call; mode PATH_AUTO,
    PATH_SEPARATE, PATH_FUSED (one cooperative launch), PATH_REPLICATED (one
    launch, routing repeated per block) or PATH_CHAINED (top-k with chunk
    ranks, a scan, the expand placing its own copies).  -> (topk_idx, topk_w,
    counts, offsets, pos, sorted_src, q, sf)."""
    _dev(scores, "scores", torch.float32)
    _dev(x, "x", torch.bfloat16)
    T, E = scores.shape
    H = x.shape[1]
    R = T * k
    idx, w = _empty((T, k), torch.int32, x), _empty((T, k), torch.float32, x)
    counts, offsets = _empty((E,), torch.int32, x), _empty((E + 1,), torch.int32, x)
    pos, src = _empty((T, k), torch.int32, x), _empty((R,), torch.int32, x)
    q, sf = (out if out is not None else
             (_empty((R, H), torch.uint8, x), _empty((R, H // GROUP), torch.float32, x)))
    if workspace is None:
        workspace = route_expand_cast_workspace(T, E, k, x)
    rc = lib().moe_route_expand_cast_fp8(_ptr(scores), T, E, k, _ptr(x), H, _ptr(idx), _ptr(w),
                                         _ptr(counts), _ptr(offsets), _ptr(pos), _ptr(src),
                                         _ptr(q), _ptr(sf), _ptr(workspace), workspace.numel(),
                                         mode, GROUP, _stream(stream))
    _check(rc, "moe_route_expand_cast_fp8")
    return idx, w, counts, offsets, pos, src, q, sf


CVT_E4M3, CVT_E2M1 = 0, 1


def debug_cvt(values: torch.Tensor, fmt: int, out=None, stream=None) -> torch.Tensor:
    """The device's f32 -> E4M3 / E2M1 conversion of every value (one code
    per byte), as the cast kernels convert; for tests."""
    _dev(values, "values", torch.float32)
    out = out if out is not None else _empty(values.shape, torch.uint8, values)
    _check(lib().moe_debug_cvt(fmt, _ptr(values), _ptr(out), values.numel(), _stream(stream)),
           "moe_debug_cvt")
    return out


def debug_set(key: int, value: int) -> None:
    _check(lib().moe_debug_set(key, int(value)), "moe_debug_set")


def expand_cast_fp8_ex_workspace_bytes(T: int, H: int, sf_flags: int) -> int:
    return int(lib().moe_expand_cast_fp8_ex_workspace_bytes(T, H, sf_flags))


def expand_cast_fp8_ex(x: torch.Tensor, pos: torch.Tensor, num_rows: int | None = None, *,
                       sorted_src=None, sf_flags: int = 0, sf_ld: int | None = None, out=None,
                       out_sf=None, workspace=None, stream=None):
    """expand_cast_fp8 with scale options (SF_COLMAJOR, SF_POW2, SF_UE8M0) and
    an optional zero-fill of the rows whose sorted_src entry is negative.
    workspace: None (direct scale stores), True (allocate one), or a uint8
    CUDA tensor; used with a column-major layout and sorted_src to write the
    scales in whole lines (sorted_src must be pos's inverse)."""
    _dev(x, "x", torch.bfloat16)
    _dev(pos, "pos", torch.int32)
    T, H = x.shape
    k = pos.shape[1]
    if sorted_src is not None:
        _dev(sorted_src, "sorted_src", torch.int32)
    R = (T * k if sorted_src is None else sorted_src.shape[0]) if num_rows is None else int(num_rows)
    if sf_ld is None and (sf_flags & SF_COLMAJOR):
        sf_ld = (R + 3) // 4 * 4
    q = out if out is not None else _empty((R, H), torch.uint8, x)
    _dev(q, "out", torch.uint8, (R, H))
    if out_sf is None:
        out_sf, sf_ld = sf_empty(R, H // GROUP, sf_flags, sf_ld, x)
    if out_sf.device.type != "cuda" or not out_sf.is_contiguous():
        raise ValueError("out_sf must be a contiguous CUDA tensor")
    if workspace is True:
        n = expand_cast_fp8_ex_workspace_bytes(T, H, sf_flags)
        workspace = _empty((n,), torch.uint8, x) if n > 0 else None
    ws_bytes = 0 if workspace is None else workspace.numel()
    rc = lib().moe_expand_cast_fp8_ex(_ptr(x), T, H, k, _ptr(pos), _ptr(sorted_src), R, _ptr(q),
                                      _ptr(out_sf), sf_flags, int(sf_ld or R), _ptr(workspace),
                                      ws_bytes, GROUP, _stream(stream))
    _check(rc, "moe_expand_cast_fp8_ex")
    return q, out_sf


def expand_cast_fp4(x: torch.Tensor, pos: torch.Tensor, num_rows: int | None = None, *,
                    group: int = 32, sorted_src=None, sf_flags: int = 0, sf_ld: int | None = None,
                    out=None, out_sf=None, workspace=None, stream=None):
    """Expand + per-group FP4 E2M1 cast -> (q [R, H/2] packed uint8, scales in
    the flagged layout).  workspace: None, True (allocate) or a uint8 CUDA
    tensor, for column-major scales written from sorted_src."""
    _dev(x, "x", torch.bfloat16)
    _dev(pos, "pos", torch.int32)
    T, H = x.shape
    k = pos.shape[1]
    if sorted_src is not None:
        _dev(sorted_src, "sorted_src", torch.int32)
    R = (T * k if sorted_src is None else sorted_src.shape[0]) if num_rows is None else int(num_rows)
    if sf_ld is None and (sf_flags & SF_COLMAJOR):
        sf_ld = (R + 3) // 4 * 4
    q = out if out is not None else _empty((R, H // 2), torch.uint8, x)
    _dev(q, "out", torch.uint8, (R, H // 2))
    if out_sf is None:
        out_sf, sf_ld = sf_empty(R, H // group, sf_flags, sf_ld, x)
    if workspace is True:
        n = int(lib().moe_expand_cast_fp4_workspace_bytes(T, H, group, sf_flags))
        workspace = _empty((n,), torch.uint8, x) if n > 0 else None
    ws_bytes = 0 if workspace is None else workspace.numel()
    rc = lib().moe_expand_cast_fp4(_ptr(x), T, H, k, _ptr(pos), _ptr(sorted_src), R, _ptr(q),
                                   _ptr(out_sf), sf_flags, int(sf_ld or R), _ptr(workspace),
                                   ws_bytes, group, _stream(stream))
    _check(rc, "moe_expand_cast_fp4")
    return q, out_sf


def swiglu_cast_fp4(x: torch.Tensor, *, group: int = 32, clamp: float | None = None, weights=None,
                    clamp_count=None, sf_flags: int = 0, sf_ld: int | None = None, out=None,
                    out_sf=None, stream=None):
    """SwiGLU (optional clamp, per-row weight, clamp counter) then the
    per-group FP4 E2M1 cast -> (q [M, N/2] packed uint8, scales)."""
    _dev(x, "x", torch.bfloat16)
    M, N2 = x.shape
    N = N2 // 2
    if weights is not None:
        _dev(weights, "weights", torch.float32, (M,))
    if clamp_count is not None:
        _dev(clamp_count, "clamp_count", torch.int64, (1,))
    if sf_ld is None and (sf_flags & SF_COLMAJOR):
        sf_ld = (M + 3) // 4 * 4
    q = out if out is not None else _empty((M, N // 2), torch.uint8, x)
    _dev(q, "out", torch.uint8, (M, N // 2))
    if out_sf is None:
        out_sf, sf_ld = sf_empty(M, N // group, sf_flags, sf_ld, x)
    rc = lib().swiglu_cast_fp4(_ptr(x), M, N, _ptr(q), _ptr(out_sf), sf_flags, int(sf_ld or M),
                               int(clamp is not None), float(clamp or 0.0), _ptr(weights),
                               _ptr(clamp_count), group, _stream(stream))
    _check(rc, "swiglu_cast_fp4")
    return q, out_sf


def swiglu_cast_fp8_ex(x: torch.Tensor, *, clamp: float | None = None, weights=None,
                       clamp_count=None, sf_flags: int = 0, sf_ld: int | None = None, out=None,
                       out_sf=None, stream=None):
    """SwiGLU with optional clamp, per-row weight and clamp counter (an int64
    CUDA tensor of one element, added to), then the cast with scale options."""
    _dev(x, "x", torch.bfloat16)
    M, N2 = x.shape
    N = N2 // 2
    if weights is not None:
        _dev(weights, "weights", torch.float32, (M,))
    if clamp_count is not None:
        _dev(clamp_count, "clamp_count", torch.int64, (1,))
    if sf_ld is None and (sf_flags & SF_COLMAJOR):
        sf_ld = (M + 3) // 4 * 4
    q = out if out is not None else _empty((M, N), torch.uint8, x)
    _dev(q, "out", torch.uint8, (M, N))
    if out_sf is None:
        out_sf, sf_ld = sf_empty(M, N // GROUP, sf_flags, sf_ld, x)
    rc = lib().swiglu_cast_fp8_ex(_ptr(x), M, N, _ptr(q), _ptr(out_sf), sf_flags, int(sf_ld or M),
                                  int(clamp is not None), float(clamp or 0.0), _ptr(weights),
                                  _ptr(clamp_count), GROUP, _stream(stream))
    _check(rc, "swiglu_cast_fp8_ex")
    return q, out_sf


def expand_cast_fp8(x: torch.Tensor, pos: torch.Tensor, num_rows: int | None = None, *,
                    out=None, out_sf=None, stream=None):
    """Per-token E4M3 cast (one fp32 scale per 128 channels) written to the
    rows pos[t, j] of the expert-sorted buffers.

    x [T, H] bfloat16, pos [T, k] int32 -> (out [R, H] uint8 E4M3 codes,
    out_sf [R, H/128] float32); R = num_rows (default T*k)."""
    _dev(x, "x", torch.bfloat16)
    _dev(pos, "pos", torch.int32)
    T, H = x.shape
    k = pos.shape[1]
    if pos.shape[0] != T:
        raise ValueError("pos must have one row per token")
    R = T * k if num_rows is None else int(num_rows)
    q = out if out is not None else _empty((R, H), torch.uint8, x)
    sf = out_sf if out_sf is not None else _empty((R, H // GROUP), torch.float32, x)
    _dev(q, "out", torch.uint8, (R, H))
    _dev(sf, "out_sf", torch.float32, (R, H // GROUP))
    rc = lib().moe_expand_cast_fp8(_ptr(x), T, H, k, _ptr(pos), R, _ptr(q), _ptr(sf), GROUP,
                                   _stream(stream))
    _check(rc, "moe_expand_cast_fp8")
    return q, sf


def swiglu_cast_fp8(x: torch.Tensor, *, out=None, out_sf=None, stream=None):
    """silu(gate) * up in fp32, then the per-128-channel E4M3 cast.

    x [M, 2N] bfloat16 (gate | up) -> (out [M, N] uint8, out_sf [M, N/128] f32)."""
    _dev(x, "x", torch.bfloat16)
    M, N2 = x.shape
    N = N2 // 2
    q = out if out is not None else _empty((M, N), torch.uint8, x)
    sf = out_sf if out_sf is not None else _empty((M, N // GROUP), torch.float32, x)
    _dev(q, "out", torch.uint8, (M, N))
    _dev(sf, "out_sf", torch.float32, (M, N // GROUP))
    rc = lib().swiglu_cast_fp8(_ptr(x), M, N, _ptr(q), _ptr(sf), GROUP, _stream(stream))
    _check(rc, "swiglu_cast_fp8")
    return q, sf


def combine(y: torch.Tensor, topk_weights: torch.Tensor, pos: torch.Tensor,
            out_dtype=torch.bfloat16, *, out=None, stream=None):
    """out[t] = sum_j w[t, j] * y[pos[t, j]], fp32 accumulation in slot order.

    y [R, H] bfloat16, w [T, k] float32, pos [T, k] int32 ->
    out [T, H] bfloat16 (or float32)."""
    _dev(y, "y", torch.bfloat16)
    _dev(topk_weights, "topk_weights", torch.float32)
    _dev(pos, "pos", torch.int32, tuple(topk_weights.shape))
    R, H = y.shape
    T, k = pos.shape
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out_dtype must be bfloat16 or float32")
    o = out if out is not None else _empty((T, H), out_dtype, y)
    _dev(o, "out", out_dtype, (T, H))
    rc = lib().moe_combine(_ptr(y), _ptr(topk_weights), _ptr(pos), T, H, k, R, _ptr(o),
                           MOE_OUT_F32 if out_dtype == torch.float32 else MOE_OUT_BF16,
                           _stream(stream))
    _check(rc, "moe_combine")
    return o


def peak_copy(src: torch.Tensor, dst: torch.Tensor, *, stream=None):
    """Device copy of src's bytes into dst (the HBM roofline probe)."""
    if src.device.type != "cuda" or dst.device.type != "cuda":
        raise ValueError("peak_copy needs CUDA tensors")
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() < n:
        raise ValueError("dst too small")
    _check(lib().moe_peak_copy(_ptr(src), _ptr(dst), n, _stream(stream)), "moe_peak_copy")


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error bits."""
    bits = ctypes.c_uint32(0)
    rc = lib().moe_get_device_status(_stream(stream), ctypes.byref(bits))
    if rc not in (MOE_OK, MOE_ERR_DEVICE):
        _check(rc, "moe_get_device_status")
    return int(bits.value)


def launch_count() -> int:
    return int(lib().moe_kernel_launch_count())


__all__ = ["lib", "MoeError", "topk_gate", "route_map", "route_map_workspace_bytes",
           "route_map_aligned", "expand_cast_fp8_padded", "expand_cast_fp8_ex",
           "expand_cast_fp8_ex_workspace_bytes", "swiglu_cast_fp8_ex", "sf_empty",
           "route_expand_cast_fp8", "route_expand_cast_workspace", "debug_set", "debug_cvt", "expand_cast_fp4", "swiglu_cast_fp4",
           "expand_cast_fp8", "swiglu_cast_fp8", "combine", "peak_copy", "device_status",
           "launch_count", "SIGNATURES"]
