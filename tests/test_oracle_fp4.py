"""Pins of the oracle's FP4 E2M1 cast (TileKernels page, sections 3.1 and
3.2 with the float4_e2m1fn output type), against what the format definition
and the arithmetic fix: the OCP MX table of E2M1 values, round-to-nearest
with ties to the even code at every midpoint, saturation, sign symmetry, the
half-step error bound; the scale as the correctly rounded quotient of exact
rationals; the floor at clamp_min_value = 6 * 2^-126; the nibble packing on a
hand-worked row; and the expand's row copies."""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_spec_values.txt")
MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _golden():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        bits, val = line.split()
        rows.append((int(bits, 2), float(val)))
    return rows


def test_values_match_the_spec_table():
    rows = _golden()
    assert len(rows) == 16
    for code, val in rows:
        got = oracle.e2m1_value(code)
        assert got == val and np.signbit(got) == np.signbit(val), (code, got, val)


def test_every_value_encodes_to_its_code():
    for code, val in _golden():
        assert int(oracle.e2m1_encode(np.float32(val))) == code


def test_ties_go_to_the_even_code_and_neighbours_to_the_nearest():
    for i in range(7):
        lo, hi = MAGS[i], MAGS[i + 1]
        mid = np.float32((lo + hi) / 2)
        even = i if i % 2 == 0 else i + 1
        assert int(oracle.e2m1_encode(mid)) == even, (lo, hi)
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(8))
        assert int(oracle.e2m1_encode(below)) == i
        assert int(oracle.e2m1_encode(above)) == i + 1
        assert int(oracle.e2m1_encode(-mid)) == 8 | even


def test_saturation_and_sign_symmetry_on_a_dense_sweep():
    v = np.linspace(-9.0, 9.0, 72001, dtype=np.float32)
    c = oracle.e2m1_encode(v)
    assert (c[v >= 6] == 7).all() and (c[v <= -6] == 15).all()
    assert int(oracle.e2m1_encode(np.float32(np.inf))) == 7
    assert int(oracle.e2m1_encode(np.float32(-np.inf))) == 15
    pos = v > 0
    cn = oracle.e2m1_encode(-v[pos])
    assert np.array_equal(cn, c[pos] | 8)
    # monotone: codes' values never decrease along the sweep
    vals = np.array([oracle.e2m1_value(int(x)) for x in range(16)])[c]
    assert (np.diff(vals) >= 0).all()
    # within half the local gap of the input (inside the representable range)
    inside = np.abs(v) <= 6
    gaps = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0, 2.0])
    mag = np.abs(v[inside]).astype(np.float64)
    idx = np.minimum(np.searchsorted(MAGS, mag, side="right") - 1, 6)
    err = np.abs(np.abs(vals[inside]) - mag)
    assert (err <= gaps[idx] / 2 + 1e-12).all()


def test_signed_zero_and_tiny_values():
    assert int(oracle.e2m1_encode(np.float32(0.0))) == 0
    assert int(oracle.e2m1_encode(np.float32(-0.0))) == 8
    assert int(oracle.e2m1_encode(np.float32(-1e-30))) == 8
    assert int(oracle.e2m1_encode(np.float32(0.2499))) == 0


def _x(T, H, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return oracle.bf16_bits((torch.randn(T, H, generator=g) * scale).to(torch.bfloat16))


def _ident(T):
    return np.arange(T, dtype=np.int32)[:, None]


@pytest.mark.parametrize("group", [16, 32, 128])
def test_scale_is_the_correctly_rounded_quotient(group):
    xb = _x(6, 256, seed=group)
    q, sf = oracle.expand_cast_fp4(xb, _ident(6), group=group)
    x = (xb.astype(np.uint32) << 16).view(np.float32)
    G = 256 // group
    floor_v = Fraction(6) * Fraction(1, 2 ** 126)
    for t in range(6):
        for g in range(G):
            amax = max(Fraction(float(a)) for a in np.abs(x[t, g * group:(g + 1) * group]))
            exact = max(amax, floor_v) / 6
            got = Fraction(float(sf[t, g]))
            # sf is fl32(exact): no fp32 value lies strictly between them
            lo = np.nextafter(np.float32(float(got)), np.float32(0))
            hi = np.nextafter(np.float32(float(got)), np.float32(np.inf))
            assert abs(got - exact) <= abs(Fraction(float(lo)) - exact)
            assert abs(got - exact) <= abs(Fraction(float(hi)) - exact)


@pytest.mark.parametrize("group", [16, 32, 128])
def test_group_max_reaches_six_and_dequant_is_within_half_a_step(group):
    xb = _x(5, 512, seed=3 * group, scale=3.0)
    q, sf = oracle.expand_cast_fp4(xb, _ident(5), group=group)
    codes = oracle.e2m1_unpack(q)
    vals = np.array([oracle.e2m1_value(c) for c in range(16)])[codes]
    x = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    G = 512 // group
    sfx = np.repeat(sf.astype(np.float64), group, axis=1)
    for t in range(5):
        for g in range(G):
            seg = slice(g * group, (g + 1) * group)
            assert np.abs(vals[t, seg]).max() == 6.0
    scaled = np.abs(x) / sfx
    gaps = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0, 2.0])
    idx = np.minimum(np.searchsorted(MAGS, np.minimum(scaled, 6.0), side="right") - 1, 6)
    err = np.abs(vals * sfx - x)
    assert (err <= (gaps[idx] / 2 + 1e-6) * sfx).all()


def test_floor_applies_below_clamp_min_value():
    xb = oracle.bf16_bits(torch.zeros(2, 64, dtype=torch.bfloat16))
    q, sf = oracle.expand_cast_fp4(xb, _ident(2), group=32)
    assert (sf == np.float32(2.0 ** -126)).all() and (q == 0).all()


def test_nibble_packing_on_a_worked_row():
    # group max 6 -> scale 1: the values are their own codes
    row = torch.tensor([0.5, -1.0, 6.0, 0.0, 1.5, -6.0, 2.0, 3.0] * 4, dtype=torch.bfloat16)
    q, sf = oracle.expand_cast_fp4(oracle.bf16_bits(row[None]), _ident(1), group=32)
    assert sf[0, 0] == np.float32(1.0)
    assert list(q[0, :4]) == [0xA1, 0x07, 0xF3, 0x54]


def test_pow2_and_ue8m0_options():
    xb = _x(4, 256, seed=11, scale=5.0)
    _, sf = oracle.expand_cast_fp4(xb, _ident(4), group=32)
    q2, sf2 = oracle.expand_cast_fp4(xb, _ident(4), group=32, flags=oracle.SF_POW2)
    m, e = np.frexp(sf2.astype(np.float64))
    assert (m == 0.5).all() and (sf2 >= sf).all() and (sf2 < 2 * sf).all()
    qb, b = oracle.expand_cast_fp4(xb, _ident(4), group=32, flags=oracle.SF_POW2 | oracle.SF_UE8M0)
    assert np.array_equal(np.ldexp(1.0, b.astype(np.int64) - 127), sf2.astype(np.float64))
    assert np.array_equal(qb, q2)


def test_expand_copies_rows_and_zero_fills():
    T, k, H = 6, 3, 256
    xb = _x(T, H, seed=5)
    pos = np.random.default_rng(0).permutation(T * k + 4)[:T * k].astype(np.int32).reshape(T, k)
    q1, s1 = oracle.expand_cast_fp4(xb, _ident(T), group=32)
    R = T * k + 4
    src = np.full(R, -1, np.int32)
    src[pos.ravel()] = np.arange(T * k, dtype=np.int32)
    q, sf = oracle.expand_cast_fp4(xb, pos, sorted_src=src, group=32)
    for t in range(T):
        for j in range(k):
            assert np.array_equal(q[pos[t, j]], q1[t]) and np.array_equal(sf[pos[t, j]], s1[t])
    pad = src < 0
    assert (q[pad] == 0).all() and (sf[pad] == 0).all()


def test_codes_use_the_inverse_of_the_stored_scale():
    """[TK] 3.2 multiplies by the inverse of the scale.  Here amax = 125/4096,
    sf = fl32(amax / 6), and v = amax / 8: v / sf is exactly the midpoint 0.75
    (ties to even: code 2), while v * fl32(1 / sf) lies just below it (code 1).
    The cast must give code 1."""
    row = torch.zeros(32)
    row[0] = 0.030517578125
    row[1] = 0.003814697265625
    xb = oracle.bf16_bits(row.to(torch.bfloat16)[None])
    q, sf = oracle.expand_cast_fp4(xb, _ident(1), group=32)
    codes = oracle.e2m1_unpack(q)
    assert codes[0, 0] == 7 and codes[0, 1] == 1


# ---------------------------------------------------------------- SwiGLU -> FP4

def _sx(M, N, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    return oracle.bf16_bits((torch.randn(M, 2 * N, generator=g) * scale).to(torch.bfloat16))


@pytest.mark.parametrize("group", [16, 32, 128])
def test_swiglu_fp4_is_the_fp4_cast_of_the_swiglu_values(group):
    """The FP4 SwiGLU equals the FP4 cast (pinned above) of the SwiGLU values
    (pinned in the FP8 pins), fed as bf16-exact rows where possible: here the
    values are checked group by group through the scale and code definitions."""
    xb = _sx(6, 256, seed=group)
    q, sf, cnt = oracle.swiglu_cast_fp4(xb, group=group)
    assert cnt == 0
    v = oracle.swiglu_values(xb).astype(np.float64)
    codes = oracle.e2m1_unpack(q)
    vals = np.array([oracle.e2m1_value(c) for c in range(16)])[codes]
    G = 256 // group
    floor_v = 6.0 * 2.0 ** -126
    for r in range(6):
        for g in range(G):
            seg = slice(g * group, (g + 1) * group)
            amax = np.abs(v[r, seg]).max()
            assert sf[r, g] == np.float32(np.float32(max(amax, floor_v)) / np.float32(6.0))
            assert np.abs(vals[r, seg]).max() == 6.0 or amax < floor_v
    err = np.abs(vals * np.repeat(sf.astype(np.float64), group, axis=1) - v)
    assert (err <= np.repeat(sf.astype(np.float64), group, axis=1) * 1.0 + 1e-30).all()


def test_swiglu_fp4_clamp_weight_and_count_match_the_fp8_variant():
    xb = _sx(8, 256, seed=3, scale=3.0)
    w = np.linspace(0.1, 1.0, 8).astype(np.float32)
    _, _, c8 = oracle.swiglu_cast_fp8_ex(xb, clamp=2.0, weights=w)
    _, _, c4 = oracle.swiglu_cast_fp4(xb, group=32, clamp=2.0, weights=w)
    assert c4 == c8 > 0
    # a weight of 2 doubles every scale and leaves the codes
    q1, s1, _ = oracle.swiglu_cast_fp4(xb, group=32, clamp=2.0, weights=np.ones(8, np.float32))
    q2, s2, _ = oracle.swiglu_cast_fp4(xb, group=32, clamp=2.0, weights=np.full(8, 2, np.float32))
    assert np.array_equal(q1, q2) and np.array_equal(s2, 2 * s1)
