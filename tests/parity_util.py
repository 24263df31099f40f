"""Comparison rules shared by the GPU parity tests.

Bit-exact: indices, counts, offsets, pos, sorted_src, E4M3 bytes and fp32
scales of the expand cast.  Tolerances (each derived in the docstring):

* top-k weights: relative 4e-6.  Both sides form exp(s_j - s_0) / sum: the
  GPU in fp32 with expf (<= 2 ulp), the oracle in double.  The fp32
  difference s_j - s_0 carries at most 2^-24 |s_j - s_0| absolute error, so for
  score gaps up to ~30 the weight's relative error stays below
  (30 + 2 + 8 + 1) * 2^-24 ~= 2.5e-6.
* SwiGLU cast: E4M3 codes within 1 ordinal step on at most 0.1% of elements
  (the stated budget); scales within relative 2^-20 (expf differs by <= 2 ulp,
  so v and the group amax differ by a few fp32 ulps).
* combine, fp32 output: |gpu - exact| <= 1e-5 * sum_j |w_j y_j| (1e-5 relative,
  measured against the magnitude of the terms so cancellation cannot inflate
  it); fp32 accumulation of k terms errs by at most k * 2^-24 of that.
* combine, bf16 output: the round-to-nearest-even bf16 of some value within
  1e-5 * sum|w y| of the exact sum (so where the sum cancels to far below the
  terms, several bf16 steps of the small result can lie inside the tolerance).
"""
from __future__ import annotations

import numpy as np

W_RTOL = 4e-6
SWIGLU_SF_RTOL = 2.0 ** -20
SWIGLU_MISMATCH_FRAC = 1e-3
COMBINE_RTOL = 1e-5


def fp8_ordinal(codes: np.ndarray) -> np.ndarray:
    """E4M3 bytes as signed integers ordered like their values (+-0 -> 0)."""
    c = codes.astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def bf16_ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def assert_equal(gpu, ref, what: str):
    gpu = np.asarray(gpu)
    ref = np.asarray(ref)
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    if not np.array_equal(gpu, ref):
        bad = np.argwhere(gpu != ref)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} of {gpu.size} differ; first at {i}: "
                             f"gpu={gpu[i]!r} oracle={ref[i]!r}")


def assert_f32_bits_equal(gpu, ref, what: str):
    assert_equal(np.ascontiguousarray(gpu, np.float32).view(np.uint32),
                 np.ascontiguousarray(ref, np.float32).view(np.uint32), what)


def assert_weights_close(gpu, ref, what="topk_weights"):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    lim = W_RTOL * np.abs(ref) + 1e-30
    if not (err <= lim).all():
        i = np.unravel_index(np.argmax(err / lim), err.shape)
        raise AssertionError(f"{what}: rel err {err[i] / abs(ref[i]):.3g} at {i}")


def check_swiglu(gpu_q, gpu_sf, ref_q, ref_sf):
    """Returns the mismatch fraction; raises if outside the budget."""
    d = np.abs(fp8_ordinal(gpu_q) - fp8_ordinal(ref_q))
    assert d.max(initial=0) <= 1, f"swiglu: a code is {d.max()} steps off"
    frac = float((d != 0).mean()) if d.size else 0.0
    assert frac <= SWIGLU_MISMATCH_FRAC, f"swiglu: {frac:.4%} of codes differ"
    rel = np.abs(gpu_sf.astype(np.float64) - ref_sf) / ref_sf
    assert (rel <= SWIGLU_SF_RTOL).all(), f"swiglu: scale rel err {rel.max():.3g}"
    return frac


def check_combine_f32(gpu, ref_f32, mag):
    err = np.abs(gpu.astype(np.float64) - ref_f32.astype(np.float64))
    lim = COMBINE_RTOL * mag.astype(np.float64) + 1e-30
    if not (err <= lim).all():
        i = np.unravel_index(np.argmax(err / lim), err.shape)
        raise AssertionError(f"combine f32: err {err[i]:.3g} > {lim[i]:.3g} at {i}")


def _bf16_neighbours(bits: np.ndarray):
    """Values of the bf16 numbers just below and just above each input."""
    o = bf16_ordinal(bits)
    def from_ord(v):
        mag = np.abs(v).astype(np.uint32)
        b = np.where(v < 0, mag | 0x8000, mag).astype(np.uint16)
        return bf16_to_f32(b).astype(np.float64)
    return from_ord(o - 1), from_ord(o + 1)


def check_combine_bf16(gpu_bits, ref_bits, ref_f32, mag):
    """gpu must be the RNE bf16 of SOME value within 1e-5 * sum|w y| of the
    exact sum: the interval [exact - tol, exact + tol] must meet the set of
    reals that round to gpu's value (bounded by the midpoints to its two bf16
    neighbours).  The oracle's own bf16 (RNE of the exact sum) always passes."""
    gpu_bits = np.asarray(gpu_bits, np.uint16)
    ref_bits = np.asarray(ref_bits, np.uint16)
    same = gpu_bits == ref_bits
    if same.all():
        return 0
    g = bf16_to_f32(gpu_bits).astype(np.float64)
    lo_n, hi_n = _bf16_neighbours(gpu_bits)
    lo_mid, hi_mid = (g + lo_n) / 2, (g + hi_n) / 2
    exact = ref_f32.astype(np.float64)
    tol = COMBINE_RTOL * mag.astype(np.float64) + 1e-30
    ok = same | ((lo_mid <= exact + tol) & (hi_mid >= exact - tol))
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError(f"combine bf16: gpu {gpu_bits[i]:#06x} oracle {ref_bits[i]:#06x} "
                             f"(exact {ref_f32[i]!r}, tol {tol[i]:.3g}) at {i}")
    return int((~same).sum())


SF_COLMAJOR, SF_POW2, SF_UE8M0 = 0x1, 0x2, 0x4


def sf_rows(sf, flags: int, rows: int, G: int) -> np.ndarray:
    """Scales of a flagged layout as f32 [rows, G] (UE8M0 bytes decoded to
    2^(byte - 127))."""
    sf = np.asarray(sf)
    if flags & SF_UE8M0:
        if flags & SF_COLMAJOR:
            words, ld, _ = sf.shape
            b = sf.transpose(1, 0, 2).reshape(ld, 4 * words)[:rows, :G]
        else:
            b = sf.reshape(rows, G)
        return np.ldexp(1.0, b.astype(np.int64) - 127).astype(np.float32)
    if flags & SF_COLMAJOR:
        return np.ascontiguousarray(sf[:, :rows].T, np.float32)
    return np.asarray(sf, np.float32).reshape(rows, G)


def fp4_ordinal(packed: np.ndarray) -> np.ndarray:
    """Packed E2M1 bytes [..., n/2] -> signed ordinals [..., n] (+-0 -> 0)."""
    b = np.asarray(packed, dtype=np.uint8)
    c = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.int32)
    c[..., 0::2] = b & 0xF
    c[..., 1::2] = b >> 4
    mag = c & 7
    return np.where(c & 8, -mag, mag)


def check_swiglu_opts(gpu_q, gpu_sf, ref_q, ref_sf, ref_sf_plain, flags: int, rows: int,
                      ordinal=fp8_ordinal):
    """SwiGLU with scale options.  Without POW2, check_swiglu on the decoded
    scales.  With POW2 the scale is a step function of the group amax: where a
    few-ulp difference in amax straddles a power of two the two sides pick
    scales a factor 2 apart.  Such groups must be rare (<= 0.1%), exactly a
    factor 2 apart, and the oracle's unrounded scale (ref_sf_plain, [rows, G])
    must sit within 2^-20 of the smaller one; every other group obeys the
    1-step / 0.1% code rule with identical scales."""
    G = ref_sf_plain.shape[1]
    gs = sf_rows(gpu_sf, flags, rows, G).astype(np.float64)
    rs = sf_rows(ref_sf, flags, rows, G).astype(np.float64)
    og, orf = ordinal(gpu_q), ordinal(ref_q)
    if not flags & SF_POW2:
        d = np.abs(og - orf)
        assert d.max(initial=0) <= 1, f"swiglu: a code is {d.max()} steps off"
        frac = float((d != 0).mean()) if d.size else 0.0
        assert frac <= SWIGLU_MISMATCH_FRAC, f"swiglu: {frac:.4%} of codes differ"
        rel = np.abs(gs - rs) / rs
        assert (rel <= SWIGLU_SF_RTOL).all(), f"swiglu: scale rel err {rel.max():.3g}"
        return frac
    diff = gs != rs
    if diff.any():
        assert diff.mean() <= SWIGLU_MISMATCH_FRAC, f"{diff.mean():.4%} of pow2 scales differ"
        lo = np.minimum(gs, rs)[diff]
        assert (np.maximum(gs, rs)[diff] == 2 * lo).all(), "pow2 scales differ by more than 2x"
        plain = ref_sf_plain.astype(np.float64)[diff]
        assert (np.abs(plain - lo) <= 2.0 ** -20 * plain).all(), "pow2 scale off a boundary"
    keep = np.repeat(~diff, og.shape[1] // G, axis=1)
    d = np.abs(og - orf)[keep]
    assert d.max(initial=0) <= 1, f"swiglu pow2: a code is {d.max()} steps off"
    frac = float((d != 0).mean()) if d.size else 0.0
    assert frac <= SWIGLU_MISMATCH_FRAC, f"swiglu pow2: {frac:.4%} of codes differ"
    return frac
