"""Seeded random sweep over shapes and options, every op through the C ABI
against the oracle: shapes the fixed parity cases do not name (odd T, E not a
power of two, every k, H across the kernel forms, all scale layouts, every
FP4 group size, padded alignments, decode shapes on the fused and replicated
paths, and the chained form).  Each case is small enough for the oracle to finish at once."""
import os

import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops, workloads
from tests.parity_util import (assert_equal, assert_f32_bits_equal, assert_weights_close,
                               check_combine_f32, check_swiglu_opts, fp4_ordinal)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
# MOE_FUZZ_CASES widens the sweep (each case has its own seed); 24 by default
CASES = int(os.environ.get("MOE_FUZZ_CASES", "24"))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from moe_routing_precision_gb300 import _build
    _build.build()
    oracle.build()
    torch.cuda.set_device(0)
    assert ops.device_status() == 0
    yield
    assert ops.device_status() == 0


def np_(t):
    return t.detach().cpu().numpy()


def _raw(t):
    return np.ascontiguousarray(np_(t)).view(np.uint8)


def _shape(rng):
    E = int(rng.choice([33, 64, 100, 128, 200, 256, 384, 1024]))
    k = int(rng.integers(1, min(E, 32) + 1))
    T = int(rng.integers(1, 700))
    return T, E, k


@pytest.mark.parametrize("case", range(CASES))
def test_route_chain(case):
    rng = np.random.default_rng(1000 + case)
    T, E, k = _shape(rng)
    H = 128 * int(rng.integers(1, 21))
    ties = bool(rng.integers(0, 2))
    inp = workloads.random_small(T, E, k, H, seed=case, ties=ties, zero_groups=True)
    s, x = inp["scores"], inp["x"]
    idx, w = ops.topk_gate(s.to(DEV), k)
    o_idx, o_w = oracle.topk_gate(s.numpy(), k)
    assert_equal(np_(idx), o_idx, "idx")
    assert_weights_close(np_(w), o_w)
    align = int(rng.choice([1, 2, 8, 64, 128] if E <= 256 else [1, 2, 16]))
    if align == 1:
        counts, offsets, pos, src = ops.route_map(idx, E)
        o_c, o_o, o_p, o_s = oracle.route_map(o_idx, E)
    else:
        counts, offsets, pos, src = ops.route_map_aligned(idx, E, align)
        o_c, o_o, o_p, o_s = oracle.route_map_aligned(o_idx, E, align)
    for a, b, n in ((counts, o_c, "counts"), (offsets, o_o, "offsets"), (pos, o_p, "pos"),
                    (src, o_s, "sorted_src")):
        assert_equal(np_(a), b, n)
    flags = int(rng.choice([0, 1, 2, 3, 6, 7]))
    R = src.shape[0]
    ld = (R + 3) // 4 * 4 + 4 * int(rng.integers(0, 3)) if flags & ops.SF_COLMAJOR else None
    sf0, ld = oracle.sf_buffer(R, H // 128, flags, ld)
    sf = torch.from_numpy(sf0.copy()).to(DEV)
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    staged = bool(rng.integers(0, 2))
    ops.expand_cast_fp8_ex(x.to(DEV), pos, sorted_src=src, sf_flags=flags, sf_ld=ld, out=q,
                           out_sf=sf, workspace=True if staged else None)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp8_ex(oracle.bf16_bits(x), o_p, sorted_src=o_s, flags=flags,
                                          ld=ld)
    assert_equal(np_(q), o_q, f"q flags={flags}")
    assert_equal(_raw(sf), np.ascontiguousarray(o_sf).view(np.uint8), f"sf flags={flags}")
    # combine over the padded or plain layout
    y = torch.randn(R, H, generator=torch.Generator().manual_seed(case)).to(torch.bfloat16)
    out = ops.combine(y.to(DEV), w, pos, torch.float32)
    o32, _, mag = oracle.combine(oracle.bf16_bits(y), o_w, o_p)
    check_combine_f32(np_(out), o32, mag)


@pytest.mark.parametrize("case", range(CASES))
def test_fp4_and_swiglu(case):
    rng = np.random.default_rng(2000 + case)
    group = int(rng.choice([16, 32, 64, 128]))
    H = 32 * int(rng.integers(1, 200))
    H -= H % group
    H = max(H, group if group >= 32 else 32)
    T, k = int(rng.integers(1, 300)), int(rng.integers(1, 9))
    x = workloads.random_small(T, 16, min(k, 16), H, seed=case, zero_groups=H % 128 == 0)["x"]
    R = T * k + int(rng.integers(0, 9))
    pos = torch.from_numpy(rng.permutation(R)[:T * k].astype(np.int32).reshape(T, k))
    pos[rng.random((T, k)) < 0.1] = -1
    flags = int(rng.choice([0, 2, 6]))
    sf0, ld = oracle.sf_buffer(R, H // group, flags, None)
    sf = torch.from_numpy(sf0.copy()).to(DEV)
    q = torch.full((R, H // 2), 0xAB, dtype=torch.uint8, device=DEV)
    ops.expand_cast_fp4(x.to(DEV), pos.to(DEV), R, group=group, sf_flags=flags, out=q, out_sf=sf)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp4(oracle.bf16_bits(x), pos.numpy(), num_rows=R, group=group,
                                       flags=flags)
    assert_equal(np_(q), o_q, f"fp4 q group={group}")
    assert_equal(_raw(sf), np.ascontiguousarray(o_sf).view(np.uint8), "fp4 sf")
    # SwiGLU, FP8 or FP4 output, random variant
    M = int(rng.integers(1, 400))
    N = 128 * int(rng.integers(1, 17))
    xs = (torch.randn(M, 2 * N, generator=torch.Generator().manual_seed(case)) * 2).to(torch.bfloat16)
    clamp = float(rng.choice([0.5, 2.0, 7.0])) if rng.integers(0, 2) else None
    wts = torch.rand(M, generator=torch.Generator().manual_seed(case + 1)) if rng.integers(0, 2) else None
    sflags = int(rng.choice([0, 1, 2, 7]))
    # the clamp count half of the time (its own generator, so the draws above
    # and below stay those of the case)
    use_cnt = bool(np.random.default_rng(3000 + case).integers(0, 2))
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    cnt_arg = cnt if use_cnt else None
    xb = oracle.bf16_bits(xs)
    wn = None if wts is None else wts.numpy()
    wd = None if wts is None else wts.to(DEV)
    if rng.integers(0, 2):
        g4 = int(rng.choice([16, 32, 64, 128]))
        q4, sf4 = ops.swiglu_cast_fp4(xs.to(DEV), group=g4, clamp=clamp, weights=wd,
                                      clamp_count=cnt_arg, sf_flags=sflags)
        o_q4, o_sf4, o_cnt = oracle.swiglu_cast_fp4(xb, group=g4, clamp=clamp, weights=wn,
                                                    flags=sflags, ld=(M + 3) // 4 * 4 if sflags & 1 else None)
        _, o_plain, _ = oracle.swiglu_cast_fp4(xb, group=g4, clamp=clamp, weights=wn)
        check_swiglu_opts(np_(q4), np_(sf4), o_q4, o_sf4, o_plain, sflags, M, ordinal=fp4_ordinal)
    else:
        q8, sf8 = ops.swiglu_cast_fp8_ex(xs.to(DEV), clamp=clamp, weights=wd,
                                         clamp_count=cnt_arg, sf_flags=sflags)
        o_q8, o_sf8, o_cnt = oracle.swiglu_cast_fp8_ex(xb, clamp=clamp, weights=wn, flags=sflags,
                                                       ld=(M + 3) // 4 * 4 if sflags & 1 else None)
        _, o_plain, _ = oracle.swiglu_cast_fp8_ex(xb, clamp=clamp, weights=wn)
        check_swiglu_opts(np_(q8), np_(sf8), o_q8, o_sf8, o_plain, sflags, M)
    assert int(cnt.item()) == (o_cnt if use_cnt else 0)
    assert ops.device_status() == 0


@pytest.mark.parametrize("case", range(CASES // 2))
@pytest.mark.parametrize("mode", ["fused", "replicated", "chained"])
def test_decode_paths(case, mode):
    rng = np.random.default_rng(3000 + case)
    E = int(rng.choice([40, 64, 96, 128, 200, 256]))
    k = int(rng.integers(1, min(E, 32) + 1))
    T = int(rng.integers(1, max(2, min(2048, 16384 // k))))
    H = 128 * int(rng.integers(1, 33))
    if mode == "replicated" and case % 3 == 0:
        T = int(rng.integers(1, 33))          # the one-launch form
    inp = workloads.random_small(T, E, k, H, seed=case, ties=bool(rng.integers(0, 2)))
    s, x = inp["scores"], inp["x"]
    if mode == "chained":
        H = 512 * int(rng.integers(1, 9))     # the chained form's H / 128 % 4 == 0
        if case % 2 == 0:
            T = int(rng.integers(2049, 40000))   # past the decode sizes, across chunk sizes
    path = {"fused": ops.PATH_FUSED, "replicated": ops.PATH_REPLICATED,
            "chained": ops.PATH_CHAINED}[mode]
    try:
        res = ops.route_expand_cast_fp8(s.to(DEV), x.to(DEV), k, mode=path)
    except ops.MoeError as e:               # a shape outside the form's limits
        assert e.rc == ops.MOE_ERR_UNSUPPORTED
        pytest.skip(f"shape outside the {mode} form")
    assert ops.device_status() == 0
    o_idx, o_w = oracle.topk_gate(s.numpy(), k)
    o_c, o_o, o_p, o_s = oracle.route_map(o_idx, E)
    o_q, o_sf = oracle.expand_cast_fp8(oracle.bf16_bits(x), o_p)
    for a, b in ((res[0], o_idx), (res[2], o_c), (res[3], o_o), (res[4], o_p), (res[5], o_s),
                 (res[6], o_q)):
        assert_equal(np_(a), b, "decode")
    assert_weights_close(np_(res[1]), o_w)
    assert_f32_bits_equal(np_(res[7]), o_sf, "decode sf")
