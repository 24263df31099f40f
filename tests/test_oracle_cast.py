"""Pins of the oracle's per-token FP8 cast, expand, SwiGLU and combine.

Cast (TileKernels page, 3.1-3.2): the scale is the correctly rounded fp32 of
max(amax, 1e-4)/448 (checked in exact rational arithmetic), every group with
amax >= 1e-4 reaches the E4M3 maximum 448, every element dequantises within
half an E4M3 step (plus the fp32 product rounding), groups are independent, and
a hand-worked group gives the expected codes.  Expand (2.2): copies land at pos
and nowhere else.  SwiGLU (3.3): numpy float64 silu(g) * u, limits g -> +-inf,
g = 0.  Combine ("CuTeDSL at Perplexity", combine): one-hot weights are the
identity, numpy float64 gather-sum, equal weights over equal rows.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _bf16(x):
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)


def _bits(x):
    return oracle.bf16_bits(_bf16(x))


def _f32_round(fr: Fraction) -> float:
    """Correctly rounded float32 of a positive normal-range rational (RNE)."""
    e = fr.numerator.bit_length() - fr.denominator.bit_length()
    if Fraction(2) ** e > fr:
        e -= 1
    quantum = Fraction(2) ** (e - 23)
    q = fr / quantum
    r = q.numerator // q.denominator
    rem = q - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    return float(r * quantum)


def _spacing(m):
    """E4M3 step at magnitude m (format definition: 3 mantissa bits, min
    normal 2^-6, subnormal step 2^-9)."""
    m = np.asarray(m, np.float64)
    out = np.full(m.shape, 2.0 ** -9)
    big = m >= 2.0 ** -6
    out[big] = 2.0 ** (np.floor(np.log2(m[big])) - 3)
    return out


def _x_random(T, H, seed, scale_mix=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g)
    if scale_mix:
        x *= 10.0 ** torch.randint(-6, 4, (T, H // 128, 1), generator=g).repeat_interleave(128, 1).reshape(T, H).float()
    return x.to(torch.bfloat16)


def test_scale_is_correctly_rounded_and_group_reaches_448():
    x = _x_random(64, 1024, 0)
    q, sf = oracle.per_token_cast(oracle.bf16_bits(x))
    xf = x.float().numpy().reshape(64, 8, 128)
    amax = np.abs(xf).max(axis=2)
    floor = Fraction(float(np.float32(1e-4)))
    for t in range(64):
        for g in range(8):
            a = max(Fraction(float(amax[t, g])), floor)
            assert float(sf[t, g]) == _f32_round(a / 448), (t, g)
    mags = (q.reshape(64, 8, 128) & 0x7F).max(axis=2)
    assert (mags[amax >= 1e-4] == 0x7E).all()


def test_dequantised_values_within_half_step():
    x = _x_random(32, 2048, 1)
    q, sf = oracle.per_token_cast(oracle.bf16_bits(x))
    xf = x.float().numpy().astype(np.float64).reshape(32, 16, 128)
    dq = oracle.e4m3_decode_fast(q).reshape(32, 16, 128)
    s = sf.astype(np.float64)[:, :, None]
    err = np.abs(dq * s - xf)
    m = np.maximum(np.abs(dq), np.abs(xf) / s)
    bound = 0.5 * _spacing(m) * s + np.abs(xf) * 2.0 ** -22
    assert (err <= bound).all()
    # signs agree (zero allowed)
    assert (np.sign(dq) * np.sign(xf) >= 0).all()


def test_zero_and_tiny_groups_use_the_floor():
    x = np.zeros((2, 256), np.float32)
    x[0, 5] = -0.0
    x[1, :128] = 3e-6           # below the 1e-4 floor
    x[1, 128:] = -2.0e-5
    q, sf = oracle.per_token_cast(_bits(x))
    floor_sf = np.float32(np.float32(1e-4) / np.float32(448.0))
    assert (sf == floor_sf).all()
    assert (q[0] & 0x7F == 0).all()
    # 3e-6 (as bf16) / (1e-4/448): about 13.4 -> 13 or 14, never the group max
    assert (q[1, :128] & 0x7F).max() < 0x7E and (q[1, 128:] >= 0x80).all()


def test_hand_worked_group():
    # amax = 1: sf = fl32(1/448) = 0x3B124925, sf_inv = fl32(1/sf) = 447.99997
    # 1.0   -> 447.99997 -> nearest E4M3 448          = 0x7E
    # -0.5  -> -223.99998 -> -224 = -(1.75 * 2^7)     = 0xF6
    # 0.25  -> 111.99999 -> 112 = 1.75 * 2^6          = 0x6E
    # 2^-7  -> 3.4999998 -> 3.5 = 1.75 * 2^1          = 0x46
    # 0.0   -> 0                                       = 0x00
    x = np.zeros((1, 128), np.float32)
    x[0, :5] = [1.0, -0.5, 0.25, 2.0 ** -7, 0.0]
    q, sf = oracle.per_token_cast(_bits(x))
    assert int(np.float32(sf[0, 0]).view(np.uint32)) == 0x3B124925
    assert list(q[0, :5]) == [0x7E, 0xF6, 0x6E, 0x46, 0x00]


def test_groups_are_independent():
    x = _x_random(4, 1024, 2)
    q, sf = oracle.per_token_cast(oracle.bf16_bits(x))
    perm = np.random.default_rng(0).permutation(8)
    xp = x.view(4, 8, 128)[:, perm].reshape(4, 1024)
    qp, sfp = oracle.per_token_cast(oracle.bf16_bits(xp))
    assert np.array_equal(qp.reshape(4, 8, 128), q.reshape(4, 8, 128)[:, perm])
    assert np.array_equal(sfp, sf[:, perm])


def test_expand_copies_rows_to_pos_only():
    x = _x_random(5, 256, 3)
    q, sf = oracle.per_token_cast(oracle.bf16_bits(x))
    pos = np.array([[3, 9], [0, -1], [7, 1], [2, 8], [6, 4]], np.int32)
    eq, esf = oracle.expand_cast_fp8(oracle.bf16_bits(x), pos, num_rows=11, fill=0xAB)
    written = set()
    for t in range(5):
        for j in range(2):
            r = pos[t, j]
            if r < 0:
                continue
            written.add(int(r))
            assert np.array_equal(eq[r], q[t]) and np.array_equal(esf[r], sf[t])
    for r in set(range(11)) - written:
        assert (eq[r] == 0xAB).all() and (esf[r] == 0).all()
    with pytest.raises(oracle.OracleError):
        oracle.expand_cast_fp8(oracle.bf16_bits(x), pos, num_rows=9)


# ---------------------------------------------------------------- SwiGLU

def test_swiglu_values_match_float64():
    g = torch.Generator().manual_seed(4)
    x = (torch.randn(64, 2 * 512, generator=g) * 4).to(torch.bfloat16)
    v = oracle.swiglu_values(oracle.bf16_bits(x))
    xf = x.double().numpy()
    gate, up = xf[:, :512], xf[:, 512:]
    ref = gate / (1.0 + np.exp(-gate)) * up
    assert (np.abs(v - ref) <= 8 * 2.0 ** -24 * np.abs(ref) + 1e-38).all()
    # the gate is the left half: swapping halves changes the values
    xs = torch.cat([x[:, 512:], x[:, :512]], 1)
    assert not np.array_equal(oracle.swiglu_values(oracle.bf16_bits(xs)), v)


def test_swiglu_limits():
    gate = np.array([0.0, 100.0, 96.0, -120.0, -200.0, 0.0], np.float32)
    up = np.array([3.0, 1.5, -2.0, 5.0, -5.0, -7.0], np.float32)
    x = np.concatenate([gate, up])[None, :]
    v = oracle.swiglu_values(_bits(x))[0]
    assert v[0] == 0.0 and v[5] == 0.0
    assert v[1] == np.float32(100.0 * 1.5) and v[2] == np.float32(96.0 * -2.0)
    assert v[3] == 0.0 and v[4] == 0.0


def test_swiglu_cast_is_cast_of_values():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(16, 2 * 1024, generator=g).to(torch.bfloat16)
    q, sf = oracle.swiglu_cast_fp8(oracle.bf16_bits(x))
    v = oracle.swiglu_values(oracle.bf16_bits(x)).astype(np.float64).reshape(16, 8, 128)
    dq = oracle.e4m3_decode_fast(q).reshape(16, 8, 128)
    s = sf.astype(np.float64)[:, :, None]
    m = np.maximum(np.abs(dq), np.abs(v) / s)
    assert (np.abs(dq * s - v) <= 0.5 * _spacing(m) * s + np.abs(v) * 2.0 ** -22).all()
    assert ((q.reshape(16, 8, 128) & 0x7F).max(axis=2) == 0x7E).all()


# ---------------------------------------------------------------- combine

def test_combine_one_hot_is_identity():
    rng = np.random.default_rng(6)
    T, k, H = 10, 4, 256
    y = _bits(rng.standard_normal((T * k, H)))
    pos = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    hot = rng.integers(0, k, T)
    w = np.zeros((T, k), np.float32)
    w[np.arange(T), hot] = 1.0
    out32, out16, _ = oracle.combine(y, w, pos)
    assert np.array_equal(out16, y[pos[np.arange(T), hot]])
    assert np.array_equal(out32.view(np.uint32) >> 16, y[pos[np.arange(T), hot]].astype(np.uint32))


def test_combine_matches_float64_gather_sum():
    rng = np.random.default_rng(7)
    T, k, H = 20, 8, 512
    yb = _bf16(rng.standard_normal((T * k, H)))
    y = oracle.bf16_bits(yb)
    pos = rng.permutation(T * k).astype(np.int32).reshape(T, k)
    w = rng.random((T, k)).astype(np.float32)
    out32, out16, mag = oracle.combine(y, w, pos)
    yf = yb.double().numpy()
    ref = np.einsum("tk,tkh->th", w.astype(np.float64), yf[pos])
    assert np.allclose(out32, ref, rtol=1.2e-7, atol=0)
    assert np.allclose(mag, np.einsum("tk,tkh->th", np.abs(w.astype(np.float64)), np.abs(yf[pos])), rtol=1e-6)
    ref16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    got16 = (out16.astype(np.uint32) << 16).view(np.float32)
    # bf16 of the exact sum vs bf16 of its float32 rounding: equal away from ties
    assert (got16 == ref16).mean() > 0.999


def test_combine_weights_summing_to_one_over_equal_rows():
    rng = np.random.default_rng(8)
    T, k, H = 16, 8, 256
    x = _bits(rng.standard_normal((T, H)))
    y = np.repeat(x, k, axis=0)                      # row t*k+j holds token t
    pos = np.arange(T * k, dtype=np.int32).reshape(T, k)
    w = np.full((T, k), 0.125, np.float32)
    _, out16, _ = oracle.combine(y, w, pos)
    assert np.array_equal(out16, x)
    s = rng.standard_normal((T, 64)).astype(np.float32)
    _, w2 = oracle.topk_gate(s, k)
    _, out16b, _ = oracle.combine(y, w2, pos)
    assert np.array_equal(out16b, x)


def test_combine_drops_negative_pos():
    y = _bits(np.ones((4, 128), np.float32))
    pos = np.array([[0, -1], [2, 3]], np.int32)
    w = np.array([[0.5, 0.5], [0.25, 0.5]], np.float32)
    out32, _, _ = oracle.combine(y, w, pos)
    assert (out32[0] == 0.5).all() and (out32[1] == 0.75).all()


def test_multiplier_is_inverse_of_stored_scale():
    """TileKernels page, 3.2: q = x * (inverse of SF), SF being the stored
    scale.  Construct groups whose amax makes fl(1/fl(amax/448)) differ from
    fl(448/amax), with an element whose code depends on which is used."""
    rng = np.random.default_rng(9)
    cands = rng.uniform(0.5, 64.0, 200000).astype(np.float32)
    cands = torch.from_numpy(cands).to(torch.bfloat16).float().numpy()  # bf16 amax
    sf = (cands / np.float32(448.0)).astype(np.float32)
    inv_a = (np.float32(1.0) / sf).astype(np.float32)
    inv_b = (np.float32(448.0) / cands).astype(np.float32)
    diff = np.nonzero(inv_a != inv_b)[0]
    assert diff.size > 0
    hits = 0
    for i in diff[:4000]:
        a = np.float32(cands[i])
        # bf16 values x in (0, a] whose scaled value lands on different codes
        xs = torch.from_numpy(np.linspace(a / 64, a, 2000, dtype=np.float32)).to(torch.bfloat16).float().numpy()
        qa = oracle.e4m3_encode((xs * inv_a[i]).astype(np.float32))
        qb = oracle.e4m3_encode((xs * inv_b[i]).astype(np.float32))
        sel = np.nonzero(qa != qb)[0]
        if sel.size == 0:
            continue
        row = np.zeros(128, np.float32)
        row[0] = a
        row[1] = xs[sel[0]]
        q, s = oracle.per_token_cast(_bits(row[None, :]))
        assert s[0, 0] == sf[i]
        assert q[0, 1] == qa[sel[0]] != qb[sel[0]]
        hits += 1
        if hits >= 20:
            break
    assert hits > 0
