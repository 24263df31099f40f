"""Pins of the oracle's E4M3FN encoder and bf16 rounding.

The encoder is pinned against (a) the OCP specification's table points, (b)
PyTorch's own CPU float32 -> float8_e4m3fn cast, exhaustively over every
non-negative float32 bit pattern below 464 (beyond that torch returns NaN,
while the method saturates), (c) the saturation closed form above 448, and (d)
sign symmetry on a random sample of negative patterns.
"""
import multiprocessing as mp
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_spec_points.txt")


def _spec_points():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            v, code = line.split()[:2]
            rows.append((float(v), int(code, 16)))
    return rows


def test_spec_points_encode_and_decode():
    for v, code in _spec_points():
        got = int(oracle.e4m3_encode(np.array([v], np.float32))[0])
        assert got == code, (v, hex(got), hex(code))
        dec = oracle.e4m3_decode(np.array([code], np.uint8))[0]
        assert dec == v and np.signbit(dec) == np.signbit(v)


def test_decode_encode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    # magnitudes strictly increase with the code
    mags = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    assert np.all(np.diff(mags) > 0) and mags[-1] == 448.0


def _torch_vs_oracle_chunk(args):
    lo, hi = args
    bits = np.arange(lo, hi, dtype=np.uint32)
    f = bits.view(np.float32)
    ours = oracle.e4m3_encode(f)
    ref = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    return int(bad.size), (int(bits[bad[0]]) if bad.size else None)


def test_encoder_exhaustive_vs_torch_nonnegative():
    """Every float32 pattern in [0, 464): 0x00000000 .. 0x43E7FFFF."""
    end = 0x43E80000  # 464.0: torch's NaN threshold for E4M3FN
    step = 1 << 25
    chunks = [(lo, min(lo + step, end)) for lo in range(0, end, step)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(8, os.cpu_count() or 1)) as pool:
        res = pool.map(_torch_vs_oracle_chunk, chunks)
    nbad = sum(r[0] for r in res)
    first = next((r[1] for r in res if r[1] is not None), None)
    assert nbad == 0, f"{nbad} mismatches, first pattern {first and hex(first)}"


def test_encoder_saturates_above_max():
    # every 4099th pattern from 448 up to +inf, plus inf itself
    bits = np.arange(0x43E00000, 0x7F800001, 4099, dtype=np.uint32)
    bits = np.concatenate([bits, np.array([0x7F800000], np.uint32)])
    f = bits.view(np.float32)
    assert np.all(oracle.e4m3_encode(f) == 0x7E)
    assert np.all(oracle.e4m3_encode(-f) == 0xFE)


def test_encoder_sign_symmetry_sample():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 0x7F800000, size=1 << 20, dtype=np.uint32)
    f = bits.view(np.float32)
    pos = oracle.e4m3_encode(f)
    neg = oracle.e4m3_encode(-f)
    assert np.array_equal(neg, pos | 0x80)


def test_encoder_ties_go_to_even_code():
    # midpoints between consecutive codes, from the format definition
    for c in range(126):
        lo, hi = Fraction(oracle.e4m3_value(c)), Fraction(oracle.e4m3_value(c + 1))
        mid = (lo + hi) / 2
        got = int(oracle.e4m3_encode(np.array([float(mid)], np.float32))[0])
        assert got == (c if c % 2 == 0 else c + 1), (c, got)


def _bf16_rne_exact(x: float) -> float:
    """Nearest bf16 (8 significant bits) to the exact rational of x, ties even."""
    fx = Fraction(x)
    if fx == 0:
        return 0.0
    a = abs(fx)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    quantum = Fraction(2) ** max(e - 7, -133)
    q = a / quantum
    r = q.numerator // q.denominator
    rem = q - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    out = float(r * quantum)
    return -out if fx < 0 else out


def test_bf16_from_double_exact_rounding():
    rng = np.random.default_rng(1)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000))
    # midpoints and near-midpoints between bf16 neighbours
    for m in range(0x3F80, 0x3F90):
        lo = np.array([m << 16], np.uint32).view(np.float32)[0]
        hi = np.array([(m + 1) << 16], np.uint32).view(np.float32)[0]
        mid = (float(lo) + float(hi)) / 2
        xs += [mid, np.nextafter(mid, 0.0), np.nextafter(mid, 10.0)]
    for x in xs:
        bits = oracle.bf16_from_double(float(x))
        got = np.array([bits << 16], np.uint32).view(np.float32)[0]
        assert float(got) == _bf16_rne_exact(float(x)), (x, hex(bits))


def test_bf16_from_double_matches_torch_on_float_inputs():
    # for values exactly representable in float32, torch's float->bf16 cast is
    # a single RNE rounding and must agree
    rng = np.random.default_rng(2)
    f = (rng.standard_normal(4096) * 100).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, ref)
