"""Pins of the oracle's cast options (TileKernels page, 3.1: round_sf and
packed UE8M0; 2.2: TMA-aligned column-major scales) and SwiGLU variants (3.3:
clamp, top-k weight, clamp count).

Every option reduces to the already-pinned plain cast when switched off;
layouts are checked as transposes / byte packings of the row-major result;
power-of-two scales against their definition via frexp; the weight by the
exact doubling invariance of the cast; the clamp against numpy float64.
"""
import numpy as np
import pytest
import torch

import oracle


def _x(T, H, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g) * scale
    x[0, :128] = 0.0                       # a group on the 1e-4 floor
    return oracle.bf16_bits(x.to(torch.bfloat16))


def _pos(T, k, seed):
    return np.random.default_rng(seed).permutation(T * k).astype(np.int32).reshape(T, k)


def test_flags_zero_is_the_plain_expand():
    x, pos = _x(20, 512, 0), _pos(20, 3, 1)
    q0, sf0 = oracle.expand_cast_fp8(x, pos)
    q1, sf1 = oracle.expand_cast_fp8_ex(x, pos)
    assert np.array_equal(q0, q1) and np.array_equal(sf0, sf1)


def test_colmajor_is_the_transpose_with_leading_dimension():
    x, pos = _x(20, 512, 2), _pos(20, 3, 3)
    q0, sf0 = oracle.expand_cast_fp8_ex(x, pos)
    q1, sf1 = oracle.expand_cast_fp8_ex(x, pos, flags=oracle.SF_COLMAJOR, ld=64)
    assert np.array_equal(q0, q1)
    assert np.array_equal(sf1[:, :60], sf0.T) and np.isnan(sf1[:, 60:]).all()


def test_pow2_scales_by_definition():
    x, pos = _x(30, 1024, 4, scale=3.0), _pos(30, 2, 5)
    _, sf0 = oracle.expand_cast_fp8_ex(x, pos)
    q2, sf2 = oracle.expand_cast_fp8_ex(x, pos, flags=oracle.SF_POW2)
    m, e = np.frexp(sf2.astype(np.float64))
    assert (m == 0.5).all()                                   # powers of two
    assert (sf2 >= sf0).all() and (sf2 < 2 * sf0).all()      # the smallest such >= sf
    mags = (q2 & 0x7F).max(axis=1)
    assert (mags <= 0x7E).all()
    # dequantised within half an E4M3 step of the input (pow2 scale is exact)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    inv = np.argsort(pos.ravel())                             # row -> (t, j)
    rows_t = inv // 2
    dq = oracle.e4m3_decode_fast(q2).reshape(60, 8, 128) * sf2[:, :, None]
    ref = xf[rows_t].reshape(60, 8, 128)
    m2 = np.abs(ref) / sf2[:, :, None]
    step = np.where(m2 >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(m2, 1e-30))) - 3), 2.0 ** -9)
    assert (np.abs(dq - ref) <= 0.5 * step * sf2[:, :, None] + 1e-30).all()


def test_ue8m0_bytes_encode_the_pow2_scale_and_pack_by_rows():
    x, pos = _x(25, 896, 6), _pos(25, 2, 7)    # G = 7: a partial packed word
    _, sfp = oracle.expand_cast_fp8_ex(x, pos, flags=oracle.SF_POW2)
    qb, b = oracle.expand_cast_fp8_ex(x, pos, flags=oracle.SF_UE8M0 | oracle.SF_POW2)
    assert np.array_equal(np.ldexp(1.0, b.astype(np.int64) - 127), sfp.astype(np.float64))
    qc, bc = oracle.expand_cast_fp8_ex(x, pos, flags=oracle.SF_UE8M0 | oracle.SF_POW2 |
                                       oracle.SF_COLMAJOR, ld=52)
    assert bc.shape == (2, 52, 4)
    unpacked = bc.transpose(1, 0, 2).reshape(52, 8)[:50, :7]
    assert np.array_equal(unpacked, b) and np.array_equal(qc, qb)


def test_zero_fill_with_options():
    T, k, H = 10, 2, 512
    x = _x(T, H, 8)
    _, _, pos, src = oracle.route_map_aligned(np.tile(np.arange(k, dtype=np.int32), (T, 1)), 4, 8)
    q, b = oracle.expand_cast_fp8_ex(x, pos, sorted_src=src, flags=oracle.SF_UE8M0 | oracle.SF_POW2)
    pad = src < 0
    assert (q[pad] == 0).all() and (b[pad] == 0).all() and not (q == 0xAB).all(axis=1).any()


# ---------------------------------------------------------------- SwiGLU

def _sx(M, N, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    return oracle.bf16_bits((torch.randn(M, 2 * N, generator=g) * scale).to(torch.bfloat16))


def test_swiglu_ex_without_options_is_the_plain_cast():
    x = _sx(20, 512, 9)
    q0, sf0 = oracle.swiglu_cast_fp8(x)
    q1, sf1, n = oracle.swiglu_cast_fp8_ex(x)
    assert np.array_equal(q0, q1) and np.array_equal(sf0, sf1) and n == 0


def test_swiglu_huge_clamp_changes_nothing():
    x = _sx(16, 256, 10)
    q0, sf0 = oracle.swiglu_cast_fp8(x)
    q1, sf1, n = oracle.swiglu_cast_fp8_ex(x, clamp=1e30)
    assert np.array_equal(q0, q1) and np.array_equal(sf0, sf1) and n == 0


def test_swiglu_clamp_against_float64_and_count():
    M, N, c = 32, 256, 1.5
    x = _sx(M, N, 11)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    g, u = xf[:, :N], xf[:, N:]
    gc, uc = np.minimum(g, c), np.clip(u, -c, c)
    ref = gc / (1 + np.exp(-gc)) * uc
    q, sf, n = oracle.swiglu_cast_fp8_ex(x, clamp=c)
    assert n == int((g > c).sum() + (np.abs(u) > c).sum())
    # the cast of values within 8 ulp of ref: compare dequantised values
    dq = oracle.e4m3_decode_fast(q).reshape(M, 2, 128) * sf[:, :, None]
    r3 = ref.reshape(M, 2, 128)
    m2 = np.abs(r3) / sf[:, :, None]
    step = np.where(m2 >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(m2, 1e-30))) - 3), 2.0 ** -9)
    assert (np.abs(dq - r3) <= (0.5 * step + 2.0 ** -18 * m2 + 1e-6) * sf[:, :, None]).all()


def test_swiglu_weight_of_two_doubles_scales_only():
    x = _sx(24, 384, 12)
    q0, sf0, _ = oracle.swiglu_cast_fp8_ex(x)
    q2, sf2, _ = oracle.swiglu_cast_fp8_ex(x, weights=np.full(24, 2.0, np.float32))
    above = sf0 > np.float32(1e-4) / np.float32(448)          # floor not active
    assert np.array_equal(sf2[above], 2 * sf0[above])
    rows = above.all(axis=1)
    assert np.array_equal(q2[rows], q0[rows])


def test_swiglu_per_row_weights_against_float64():
    M, N = 16, 256
    x = _sx(M, N, 13)
    w = np.random.default_rng(14).random(M).astype(np.float32) + 0.1
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    g, u = xf[:, :N], xf[:, N:]
    ref = g / (1 + np.exp(-g)) * u * w[:, None].astype(np.float64)
    q, sf, _ = oracle.swiglu_cast_fp8_ex(x, weights=w)
    dq = oracle.e4m3_decode_fast(q).reshape(M, 2, 128) * sf[:, :, None]
    r3 = ref.reshape(M, 2, 128)
    m2 = np.abs(r3) / sf[:, :, None]
    step = np.where(m2 >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(m2, 1e-30))) - 3), 2.0 ** -9)
    assert (np.abs(dq - r3) <= (0.5 * step + 2.0 ** -18 * m2 + 1e-6) * sf[:, :, None]).all()
