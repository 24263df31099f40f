"""CPU oracle for the MoE routing + FP8 quantisation path.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline / reference leg may import this module; the product path never
does.  It wraps ``oracle.c`` (plain single-threaded C, compiled without
fast-math and with ``-ffp-contract=off``) through ctypes over numpy arrays, and
shares nothing with the CUDA library.

Each function names the passage it follows; the C source carries the full
statement.  Pins for every function live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CC_FLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        cc = os.environ.get("CC", "gcc")
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [cc, *CC_FLAGS, _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int32
            sig = {
                "oracle_e4m3_value": (ctypes.c_double, [ctypes.c_int]),
                "oracle_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
                "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
                "oracle_e4m3_encode_array": (None, [P, i64, P]),
                "oracle_e2m1_value": (ctypes.c_double, [ctypes.c_int]),
                "oracle_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
                "oracle_e2m1_encode_array": (None, [P, i64, P]),
                "oracle_swiglu_cast_fp4": (ctypes.c_int, [P, i64, i32, i32, i32, ctypes.c_float, P,
                                                          i32, i64, P, P, P]),
                "oracle_expand_cast_fp4": (ctypes.c_int, [P, i64, i32, i32, P, P, i64, i32, i32,
                                                          i64, P, P]),
                "oracle_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
                "oracle_topk_gate": (ctypes.c_int, [P, i64, i32, i32, P, P]),
                "oracle_route_map": (ctypes.c_int, [P, i64, i32, i32, P, P, P, P]),
                "oracle_route_map_aligned": (ctypes.c_int, [P, i64, i32, i32, i32, i64, P, P, P, P]),
                "oracle_expand_cast_fp8_padded": (ctypes.c_int, [P, i64, i32, i32, P, P, i64, i32, P, P]),
                "oracle_expand_cast_fp8_ex": (ctypes.c_int, [P, i64, i32, i32, P, P, i64, i32, i32,
                                                             i64, P, P]),
                "oracle_swiglu_cast_fp8_ex": (ctypes.c_int, [P, i64, i32, i32, i32, ctypes.c_float, P,
                                                             i32, i64, P, P, P]),
                "oracle_per_token_cast": (ctypes.c_int, [P, i64, i32, i32, P, P]),
                "oracle_expand_cast_fp8": (ctypes.c_int, [P, i64, i32, i32, P, i64, i32, P, P]),
                "oracle_swiglu_values": (ctypes.c_int, [P, i64, i32, P]),
                "oracle_swiglu_cast_fp8": (ctypes.c_int, [P, i64, i32, i32, P, P]),
                "oracle_combine": (ctypes.c_int, [P, P, P, i64, i32, i32, i64, P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc == 1:
        raise OracleError(f"{what}: invalid argument")
    if rc == 2:
        raise OracleError(f"{what}: input outside the method's domain (NaN or index out of range)")
    if rc != 0:
        raise OracleError(f"{what}: rc={rc}")


def _as(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def bf16_bits(a) -> np.ndarray:
    """View a bf16 tensor/array as its uint16 bit patterns (no arithmetic)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16
            return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    return _as(a, np.uint16)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Magnitude of a 7-bit E4M3FN code (OCP FP8 format definition)."""
    return _load().oracle_e4m3_value(int(code))


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_decode(int(v)) for v in c]).reshape(np.shape(codes))


E4M3_DECODE_TABLE = None


def e4m3_decode_fast(codes: np.ndarray) -> np.ndarray:
    """Decode through a 256-entry table built from ``e4m3_decode``."""
    global E4M3_DECODE_TABLE
    if E4M3_DECODE_TABLE is None:
        E4M3_DECODE_TABLE = e4m3_decode(np.arange(256, dtype=np.uint8))
    return E4M3_DECODE_TABLE[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Round to nearest E4M3FN, ties to even code, saturating at 448."""
    v = _as(np.asarray(v, dtype=np.float32), np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (OCP Microscaling FP4 element type)."""
    return _load().oracle_e2m1_value(int(code))


def e2m1_encode(v) -> np.ndarray:
    """Round to nearest E2M1, ties to even code, saturating at 6; one code
    (0..15) per value."""
    shape = np.shape(v)
    v = _as(np.asarray(v, dtype=np.float32), np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(v), v.size, _ptr(out))
    return out.reshape(shape)


def e2m1_unpack(packed) -> np.ndarray:
    """[..., n/2] packed bytes -> [..., n] codes (element 2i = low nibble)."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def bf16_from_double(x: float) -> int:
    return int(_load().oracle_bf16_from_double(float(x)))


# --------------------------------------------------------------------------
# The five steps
# --------------------------------------------------------------------------

def topk_gate(scores, k: int, weights: bool = True):
    """TileKernels page, 2.1 Top-K Gating (+ softmax over the k selected).

    scores [T, E] float32 -> (idx [T, k] int32, w [T, k] float32 or None)."""
    s = _as(scores, np.float32)
    T, E = s.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32) if weights else None
    _check(_load().oracle_topk_gate(_ptr(s), T, E, k, _ptr(idx), _ptr(w)), "topk_gate")
    return idx, w


def route_map(topk_idx, num_experts: int):
    """CuTeDSL at Perplexity, MoE dispatch: per-expert counts, exclusive
    offsets, stable slot per routed copy and its inverse.

    -> (counts [E], offsets [E+1], pos [T, k], sorted_src [T*k]) all int32."""
    idx = _as(topk_idx, np.int32)
    T, k = idx.shape
    E = int(num_experts)
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    pos = np.empty((T, k), dtype=np.int32)
    src = np.empty(T * k, dtype=np.int32)
    _check(_load().oracle_route_map(_ptr(idx), T, E, k, _ptr(counts), _ptr(offsets),
                                    _ptr(pos), _ptr(src)), "route_map")
    return counts, offsets, pos, src


def route_map_aligned(topk_idx, num_experts: int, align: int, num_rows: int | None = None):
    """Padded expert layout: segments rounded up to `align` rows; padding
    rows and the tail up to num_rows (default T*k + E*(align-1)) have
    sorted_src = -1.  -> (counts, offsets [E+1], pos [T,k], sorted_src [num_rows])."""
    idx = _as(topk_idx, np.int32)
    T, k = idx.shape
    E = int(num_experts)
    R = T * k + E * (align - 1) if num_rows is None else int(num_rows)
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    pos = np.empty((T, k), dtype=np.int32)
    src = np.empty(R, dtype=np.int32)
    _check(_load().oracle_route_map_aligned(_ptr(idx), T, E, k, int(align), R, _ptr(counts),
                                            _ptr(offsets), _ptr(pos), _ptr(src)),
           "route_map_aligned")
    return counts, offsets, pos, src


def expand_cast_fp8_padded(x_bits, pos, sorted_src, group: int = 128, fill: int = 0xAB):
    """Expand into the padded layout, zero-filling the rows with sorted_src < 0
    (rows named by pos are written; nothing else should remain at `fill`)."""
    x = _as(x_bits, np.uint16)
    p = _as(pos, np.int32)
    src = _as(sorted_src, np.int32)
    T, H = x.shape
    k = p.shape[1]
    R = src.shape[0]
    q = np.full((R, H), fill, dtype=np.uint8)
    sf = np.full((R, H // group), np.nan, dtype=np.float32)
    _check(_load().oracle_expand_cast_fp8_padded(_ptr(x), T, H, k, _ptr(p), _ptr(src), R, group,
                                                 _ptr(q), _ptr(sf)), "expand_cast_fp8_padded")
    return q, sf


SF_COLMAJOR, SF_POW2, SF_UE8M0 = 1, 2, 4


def sf_buffer(rows: int, G: int, flags: int, ld: int | None = None):
    """An empty scale buffer of the layout `flags` names (filled with a
    sentinel: NaN for f32, 0xAB for bytes) and its leading dimension."""
    ld = rows if ld is None else ld
    if flags & SF_UE8M0:
        if flags & SF_COLMAJOR:
            return np.full((-(-G // 4), ld, 4), 0xAB, np.uint8), ld
        return np.full((rows, G), 0xAB, np.uint8), ld
    if flags & SF_COLMAJOR:
        return np.full((G, ld), np.nan, np.float32), ld
    return np.full((rows, G), np.nan, np.float32), ld


def expand_cast_fp8_ex(x_bits, pos, num_rows: int | None = None, sorted_src=None,
                       flags: int = 0, ld: int | None = None, group: int = 128, fill: int = 0xAB):
    """Expand + cast with scale options (SF_COLMAJOR, SF_POW2, SF_UE8M0) and an
    optional zero-fill of the rows with sorted_src < 0.
    -> (q [R, H] uint8, scales in the flagged layout)."""
    x = _as(x_bits, np.uint16)
    p = _as(pos, np.int32)
    T, H = x.shape
    k = p.shape[1]
    R = (T * k if sorted_src is None else len(sorted_src)) if num_rows is None else int(num_rows)
    src = None if sorted_src is None else _as(sorted_src, np.int32)
    q = np.full((R, H), fill, dtype=np.uint8)
    sf, ld = sf_buffer(R, H // group, flags, ld)
    _check(_load().oracle_expand_cast_fp8_ex(_ptr(x), T, H, k, _ptr(p), _ptr(src), R, group,
                                             int(flags), int(ld), _ptr(q), _ptr(sf)),
           "expand_cast_fp8_ex")
    return q, sf


def swiglu_cast_fp8_ex(x_bits, clamp: float | None = None, weights=None, flags: int = 0,
                       ld: int | None = None, group: int = 128):
    """SwiGLU with optional clamp and per-row weight, then the cast with scale
    options.  -> (q [M, N], scales in the flagged layout, clamp count)."""
    x = _as(x_bits, np.uint16)
    M, N2 = x.shape
    N = N2 // 2
    w = None if weights is None else _as(np.asarray(weights, np.float32), np.float32)
    q = np.empty((M, N), dtype=np.uint8)
    sf, ld = sf_buffer(M, N // group, flags, ld)
    cnt = np.zeros(1, dtype=np.uint64)
    _check(_load().oracle_swiglu_cast_fp8_ex(_ptr(x), M, N, group, int(clamp is not None),
                                             float(clamp or 0.0), _ptr(w), int(flags), int(ld),
                                             _ptr(q), _ptr(sf), _ptr(cnt)), "swiglu_cast_fp8_ex")
    return q, sf, int(cnt[0])


def expand_cast_fp4(x_bits, pos, num_rows: int | None = None, sorted_src=None, group: int = 32,
                    flags: int = 0, ld: int | None = None, fill: int = 0xAB):
    """TileKernels page, 3.1 + 3.2 + 2.2 with the FP4 output type: per-group
    E2M1 cast (max 6, clamp_min 6 * 2^-126) of each token, copied to its pos
    rows.  -> (q [R, H/2] packed uint8, scales in the flagged layout)."""
    x = _as(x_bits, np.uint16)
    p = _as(pos, np.int32)
    T, H = x.shape
    k = p.shape[1]
    R = (T * k if sorted_src is None else len(sorted_src)) if num_rows is None else int(num_rows)
    src = None if sorted_src is None else _as(sorted_src, np.int32)
    q = np.full((R, H // 2), fill, dtype=np.uint8)
    sf, ld = sf_buffer(R, H // group, flags, ld)
    _check(_load().oracle_expand_cast_fp4(_ptr(x), T, H, k, _ptr(p), _ptr(src), R, group,
                                          int(flags), int(ld), _ptr(q), _ptr(sf)),
           "expand_cast_fp4")
    return q, sf


def swiglu_cast_fp4(x_bits, group: int = 32, clamp: float | None = None, weights=None,
                    flags: int = 0, ld: int | None = None):
    """TileKernels page, 3.3 with the FP4 output type: SwiGLU (optional clamp
    and per-row weight) then the per-group E2M1 cast.  -> (q [M, N/2] packed,
    scales in the flagged layout, clamp count)."""
    x = _as(x_bits, np.uint16)
    M, N2 = x.shape
    N = N2 // 2
    w = None if weights is None else _as(np.asarray(weights, np.float32), np.float32)
    q = np.empty((M, N // 2), dtype=np.uint8)
    sf, ld = sf_buffer(M, N // group, flags, ld)
    cnt = np.zeros(1, dtype=np.uint64)
    _check(_load().oracle_swiglu_cast_fp4(_ptr(x), M, N, group, int(clamp is not None),
                                          float(clamp or 0.0), _ptr(w), int(flags), int(ld),
                                          _ptr(q), _ptr(sf), _ptr(cnt)), "swiglu_cast_fp4")
    return q, sf, int(cnt[0])


def per_token_cast(x_bits, group: int = 128):
    """TileKernels page, 3.2 per_token_cast: x [T, H] bf16 bits (uint16) ->
    (q [T, H] uint8 E4M3 codes, sf [T, H/group] float32)."""
    x = _as(x_bits, np.uint16)
    T, H = x.shape
    q = np.empty((T, H), dtype=np.uint8)
    sf = np.empty((T, H // group), dtype=np.float32)
    _check(_load().oracle_per_token_cast(_ptr(x), T, H, group, _ptr(q), _ptr(sf)), "per_token_cast")
    return q, sf


def expand_cast_fp8(x_bits, pos, num_rows: int | None = None, group: int = 128,
                    fill: int = 0):
    """TileKernels page, 3.2 + 2.2: per_token_cast then expand_to_fused.

    x [T, H] bf16 bits, pos [T, k] int32 -> (q [R, H] uint8, sf [R, G] f32).
    Rows that no pos names keep ``fill`` (bytes) / 0.0 (scales)."""
    x = _as(x_bits, np.uint16)
    p = _as(pos, np.int32)
    T, H = x.shape
    k = p.shape[1]
    R = T * k if num_rows is None else int(num_rows)
    q = np.full((R, H), fill, dtype=np.uint8)
    sf = np.zeros((R, H // group), dtype=np.float32)
    _check(_load().oracle_expand_cast_fp8(_ptr(x), T, H, k, _ptr(p), R, group, _ptr(q), _ptr(sf)),
           "expand_cast_fp8")
    return q, sf


def expand_cast_fp8_into(x_bits, pos, q, sf, group: int = 128):
    """expand_cast_fp8 writing into the caller's arrays: q [R, H] uint8 and
    sf [R, H/group] float32 (rows no pos names are left as they are).  Only
    the marshalling differs, so token shards may run in separate threads (the
    C call releases the GIL; each shard writes its own rows)."""
    x = _as(x_bits, np.uint16)
    p = _as(pos, np.int32)
    T, H = x.shape
    k = p.shape[1]
    if q.dtype != np.uint8 or sf.dtype != np.float32 or q.shape[1] != H or \
            sf.shape != (q.shape[0], H // group):
        raise TypeError("q must be uint8 [R, H] and sf float32 [R, H/group]")
    _check(_load().oracle_expand_cast_fp8(_ptr(x), T, H, k, _ptr(p), q.shape[0], group, _ptr(q),
                                          _ptr(sf)), "expand_cast_fp8")


def swiglu_values(x_bits):
    """TileKernels page, 3.3: fp32 silu(gate) * up, before the cast."""
    x = _as(x_bits, np.uint16)
    M, N2 = x.shape
    v = np.empty((M, N2 // 2), dtype=np.float32)
    _check(_load().oracle_swiglu_values(_ptr(x), M, N2 // 2, _ptr(v)), "swiglu_values")
    return v


def swiglu_cast_fp8(x_bits, group: int = 128):
    """TileKernels page, 3.3: x [M, 2N] bf16 bits -> (q [M, N], sf [M, N/group])."""
    x = _as(x_bits, np.uint16)
    M, N2 = x.shape
    N = N2 // 2
    q = np.empty((M, N), dtype=np.uint8)
    sf = np.empty((M, N // group), dtype=np.float32)
    _check(_load().oracle_swiglu_cast_fp8(_ptr(x), M, N, group, _ptr(q), _ptr(sf)), "swiglu_cast_fp8")
    return q, sf


def combine(y_bits, w, pos, num_rows: int | None = None):
    """CuTeDSL at Perplexity, combine: out[t] = sum_j w[t,j] * y[pos[t,j]].

    Returns (out_f32 [T, H] float32, out_bf16_bits [T, H] uint16,
    abs_sum [T, H] float32 = sum_j |w y|)."""
    y = _as(y_bits, np.uint16)
    wt = _as(w, np.float32)
    p = _as(pos, np.int32)
    T, k = p.shape
    H = y.shape[1]
    R = y.shape[0] if num_rows is None else int(num_rows)
    out32 = np.empty((T, H), dtype=np.float32)
    out16 = np.empty((T, H), dtype=np.uint16)
    mag = np.empty((T, H), dtype=np.float32)
    _check(_load().oracle_combine(_ptr(y), _ptr(wt), _ptr(p), T, H, k, R, _ptr(out32), _ptr(out16),
                                  _ptr(mag)), "combine")
    return out32, out16, mag


__all__ = [
    "build", "OracleError", "bf16_bits", "e4m3_value", "e4m3_decode", "e4m3_decode_fast",
    "e4m3_encode", "bf16_from_double", "topk_gate", "route_map", "route_map_aligned",
    "expand_cast_fp8_padded", "expand_cast_fp8_ex", "swiglu_cast_fp8_ex", "sf_buffer",
    "SF_COLMAJOR", "SF_POW2", "SF_UE8M0", "per_token_cast",
    "expand_cast_fp8", "swiglu_values", "swiglu_cast_fp8", "combine",
]

if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
