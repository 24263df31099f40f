"""GPU parity of the cast variants (TileKernels article, sections 2.2, 3.1 and
3.3): column-major and packed UE8M0 scales, power-of-two scales, zero-filled
padding rows, and the SwiGLU clamp, per-row weight and clamp count, each
through the C ABI against the oracle.  Expand results are bit-exact, scale
buffers included (the sentinel around the written entries must survive);
SwiGLU follows the rules in tests/parity_util.py."""
import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops, workloads
from tests.parity_util import assert_equal, check_swiglu_opts, fp4_ordinal

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FLAGS = [0, 1, 2, 3, 6, 7]     # UE8M0 always with POW2


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


def _sentinel_sf(rows, G, flags, ld):
    ref, ld = oracle.sf_buffer(rows, G, flags, ld)
    return torch.from_numpy(ref.copy()).to(DEV), ld


def _raw_equal(gpu_sf, ref_sf, what):
    g = np.ascontiguousarray(np_(gpu_sf))
    r = np.ascontiguousarray(ref_sf)
    assert_equal(g.view(np.uint8), r.view(np.uint8), what)


# ---------------------------------------------------------------- expand + cast

@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("T,H,k", [(9, 256, 2), (13, 384, 3), (40, 512, 4), (21, 7168, 8),
                                   (5, 20480, 2), (3, 17024, 2)])
def test_expand_ex_parity(flags, T, H, k):
    x = workloads.random_small(T, 16, k, H, seed=T * H + flags, zero_groups=True)["x"]
    R = T * k + 5                                   # rows no pos names stay untouched
    g = torch.Generator().manual_seed(flags + H)
    pos = torch.randperm(R, generator=g)[:T * k].to(torch.int32).view(T, k)
    pos[::4, 0] = -1                                # dropped copies
    ld = (R + 3) // 4 * 4 + 4 if flags & ops.SF_COLMAJOR else None
    G = H // 128
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sf, ld = _sentinel_sf(R, G, flags, ld)
    ops.expand_cast_fp8_ex(x.to(DEV), pos.to(DEV), R, sf_flags=flags, sf_ld=ld, out=q, out_sf=sf)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp8_ex(oracle.bf16_bits(x), pos.numpy(), num_rows=R,
                                          flags=flags, ld=ld)
    assert_equal(np_(q), o_q, f"expand_ex q flags={flags}")
    _raw_equal(sf, o_sf, f"expand_ex sf flags={flags}")


@pytest.mark.parametrize("flags,off", [(6, 0), (6, 1), (6, 4), (6, 8), (2, 0), (2, 4), (2, 16)])
@pytest.mark.parametrize("T,H,k", [(7, 512, 3), (11, 1024, 32), (9, 1536, 5), (21, 7168, 8),
                                   (6, 7168, 20), (3, 16384, 2)])
def test_expand_ex_rowmajor_scales_at_offsets(flags, off, T, H, k):
    """Row-major scales (f32 power-of-two, packed UE8M0 bytes) written into a
    buffer that starts `off` bytes into an allocation: 8-, 4- and 1-byte
    alignments for the bytes, 4 and 16 for the f32 rows, row lengths G of 4,
    8, 12, 56 and 128 entries and k up to 32 copies.  The bytes around the
    scale buffer must keep their fill."""
    x = workloads.random_small(T, 16, k, H, seed=T * H + off, zero_groups=True)["x"]
    R = T * k + 3
    g = torch.Generator().manual_seed(off + H + k)
    pos = torch.randperm(R, generator=g)[:T * k].to(torch.int32).view(T, k)
    pos[1::3, k - 1] = -1
    G = H // 128
    ref, _ = oracle.sf_buffer(R, G, flags)
    raw = np.ascontiguousarray(ref).view(np.uint8).reshape(-1)
    buf = torch.full((raw.size + off + 32,), 0x5C, dtype=torch.uint8, device=DEV)
    buf[off:off + raw.size] = torch.from_numpy(raw.copy()).to(DEV)
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    ops.expand_cast_fp8_ex(x.to(DEV), pos.to(DEV), R, sf_flags=flags, out=q,
                           out_sf=buf[off:off + raw.size])
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp8_ex(oracle.bf16_bits(x), pos.numpy(), num_rows=R,
                                          flags=flags)
    assert_equal(np_(q), o_q, "rowmajor q")
    got = np_(buf)
    assert_equal(got[off:off + raw.size], np.ascontiguousarray(o_sf).view(np.uint8).reshape(-1),
                 "rowmajor sf")
    assert (got[:off] == 0x5C).all() and (got[off + raw.size:] == 0x5C).all()


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("T,E,k,H,align", [(60, 16, 4, 512, 32), (37, 16, 2, 384, 16),
                                           (30, 8, 8, 7168, 128)])
def test_expand_ex_padded_zero_fill(flags, T, E, k, H, align):
    x = workloads.random_small(T, E, k, H, seed=T + flags, zero_groups=True)["x"]
    idx = torch.stack([torch.randperm(E, generator=torch.Generator().manual_seed(t))[:k]
                       for t in range(T)]).to(torch.int32)
    _, _, o_pos, o_src = oracle.route_map_aligned(idx.numpy(), E, align)
    pos, src = torch.from_numpy(o_pos).to(DEV), torch.from_numpy(o_src).to(DEV)
    R = src.shape[0]
    ld = (R + 3) // 4 * 4 if flags & ops.SF_COLMAJOR else None
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sf, ld = _sentinel_sf(R, H // 128, flags, ld)
    ops.expand_cast_fp8_ex(x.to(DEV), pos, sorted_src=src, sf_flags=flags, sf_ld=ld, out=q,
                           out_sf=sf)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp8_ex(oracle.bf16_bits(x), o_pos, sorted_src=o_src,
                                          flags=flags, ld=ld)
    assert_equal(np_(q), o_q, "padded ex q")
    _raw_equal(sf, o_sf, "padded ex sf")


def _route(T, E, k, align, seed):
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    if align == 1:
        _, _, pos, src = oracle.route_map(idx.numpy(), E)
    else:
        _, _, pos, src = oracle.route_map_aligned(idx.numpy(), E, align)
    return pos, src


@pytest.mark.parametrize("flags", [1, 3, 7])
@pytest.mark.parametrize("T,E,k,H,align", [(50, 16, 4, 512, 1), (37, 16, 2, 384, 16),
                                           (30, 8, 8, 7168, 128), (9, 16, 2, 20480, 1),
                                           (5, 8, 2, 17024, 4), (300, 64, 8, 1024, 1)])
def test_expand_ex_staged_colmajor(flags, T, E, k, H, align):
    """Column-major scales staged per token and written from sorted_src."""
    x = workloads.random_small(T, E, k, H, seed=T + H + flags, zero_groups=True)["x"]
    o_pos, o_src = _route(T, E, k, align, seed=T + align)
    R = o_src.size
    ld = (R + 3) // 4 * 4 + 4
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sf, ld = _sentinel_sf(R, H // 128, flags, ld)
    ops.expand_cast_fp8_ex(x.to(DEV), torch.from_numpy(o_pos).to(DEV),
                           sorted_src=torch.from_numpy(o_src).to(DEV), sf_flags=flags, sf_ld=ld,
                           out=q, out_sf=sf, workspace=True)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp8_ex(oracle.bf16_bits(x), o_pos, sorted_src=o_src,
                                          flags=flags, ld=ld)
    assert_equal(np_(q), o_q, "staged q")
    _raw_equal(sf, o_sf, "staged sf")


@pytest.mark.parametrize("flags", [1, 7])
def test_expand_ex_staged_flags_bad_sorted_src(flags):
    T, E, k, H = 20, 8, 2, 512
    x = workloads.random_small(T, E, k, H, seed=1)["x"]
    o_pos, o_src = _route(T, E, k, 1, seed=2)
    src = o_src.copy()
    src[5] = T * k + 3                              # names no routed copy
    R = src.size
    sf, ld = _sentinel_sf(R, H // 128, flags, R)
    q = torch.zeros(R, H, dtype=torch.uint8, device=DEV)
    ops.expand_cast_fp8_ex(x.to(DEV), torch.from_numpy(o_pos).to(DEV),
                           sorted_src=torch.from_numpy(src).to(DEV), sf_flags=flags, sf_ld=ld,
                           out=q, out_sf=sf, workspace=True)
    assert ops.device_status() == ops.MOE_DEVERR_POS_RANGE
    o_q, o_sf = oracle.expand_cast_fp8_ex(oracle.bf16_bits(x), o_pos, sorted_src=o_src,
                                          flags=flags, ld=ld)
    assert_equal(np_(q), o_q, "codes are written by pos")
    g_sf = np_(sf)
    if flags & ops.SF_UE8M0:
        assert (g_sf[:, 5, :] == 0).all()
        g_sf[:, 5, :] = o_sf[:, 5, :]
    else:
        assert (g_sf[:, 5] == 0).all()
        g_sf[:, 5] = o_sf[:, 5]
    assert_equal(g_sf.view(np.uint8), np.ascontiguousarray(o_sf).view(np.uint8), "other rows")


@pytest.mark.parametrize("flags", [2, 7])
def test_expand_ex_extreme_values(flags):
    H = 512
    bf = torch.finfo(torch.bfloat16)
    rows = [torch.full((H,), bf.max), torch.full((H,), -bf.tiny), torch.zeros(H),
            torch.linspace(-3e4, 3e4, H), torch.randn(H) * 1e-38]
    r = torch.randn(H)
    r[7] = 1e30
    rows.append(r)
    # amax / 448 exactly a power of two: the rounding must keep it
    rows.append(torch.full((H,), 448.0 * 2.0 ** -3))
    x = torch.stack(rows).to(torch.bfloat16)
    T = x.shape[0]
    pos = workloads.random_permutation_pos(T, 2, seed=2)
    ld = (2 * T + 3) // 4 * 4 if flags & ops.SF_COLMAJOR else None
    q, sf = ops.expand_cast_fp8_ex(x.to(DEV), pos.to(DEV), sf_flags=flags, sf_ld=ld)
    o_q, o_sf = oracle.expand_cast_fp8_ex(oracle.bf16_bits(x), pos.numpy(), flags=flags, ld=ld)
    assert_equal(np_(q), o_q, "extreme ex q")
    sf_np = np_(sf)
    if flags & ops.SF_COLMAJOR:                      # padding columns are unspecified
        sf_np, o_sf = sf_np[:, :2 * T], o_sf[:, :2 * T]
    _raw_equal(torch.from_numpy(np.ascontiguousarray(sf_np)), o_sf, "extreme ex sf")


def test_expand_ex_pos_out_of_range_flags_and_skips():
    T, k, H, R = 4, 2, 512, 8
    x = workloads.random_small(T, 16, k, H, seed=4)["x"].to(DEV)
    pos = torch.tensor([[0, 1], [2, 3], [4, 9], [5, 6]], dtype=torch.int32, device=DEV)
    sf, ld = _sentinel_sf(R, H // 128, 7, 8)
    q = torch.zeros(R, H, dtype=torch.uint8, device=DEV)
    ops.expand_cast_fp8_ex(x, pos, R, sf_flags=7, sf_ld=ld, out=q, out_sf=sf)
    assert ops.device_status() == ops.MOE_DEVERR_POS_RANGE
    assert int(q[7].sum()) == 0
    assert (np_(sf)[:, 7] == 0xAB).all()


# ---------------------------------------------------------------- SwiGLU

def _swiglu_x(M, N, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(M, 2 * N, generator=g) * scale).to(torch.bfloat16)


# (clamp, per-row weights, clamp count): with the scale flags, every option
# set the kernels specialise on (the count with and without a clamp)
VARIANTS = {"plain": (None, False, False), "count": (None, False, True),
            "weight": (None, True, False), "clamp": (2.5, False, False),
            "clamp_count": (2.5, False, True), "clamp_weight": (1.0, True, False),
            "clamp_weight_count": (1.0, True, True)}


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("M,N", [(1, 128), (7, 384), (100, 2048), (1000, 256)])
def test_swiglu_ex_parity(flags, variant, M, N):
    clamp, with_w, with_cnt = VARIANTS[variant]
    x = _swiglu_x(M, N, seed=M + N + flags)
    w = torch.rand(M, generator=torch.Generator().manual_seed(M)) if with_w else None
    ld = (M + 3) // 4 * 4 + 8 if flags & ops.SF_COLMAJOR else None
    G = N // 128
    sf, ld = _sentinel_sf(M, G, flags, ld)
    cnt = torch.full((1,), 5, dtype=torch.int64, device=DEV)    # counts are added
    q, _ = ops.swiglu_cast_fp8_ex(x.to(DEV), clamp=clamp,
                                  weights=None if w is None else w.to(DEV),
                                  clamp_count=cnt if with_cnt else None, sf_flags=flags,
                                  sf_ld=ld, out_sf=sf)
    xb = oracle.bf16_bits(x)
    wn = None if w is None else w.numpy()
    o_q, o_sf, o_cnt = oracle.swiglu_cast_fp8_ex(xb, clamp=clamp, weights=wn, flags=flags, ld=ld)
    _, o_plain, _ = oracle.swiglu_cast_fp8_ex(xb, clamp=clamp, weights=wn)
    check_swiglu_opts(np_(q), np_(sf), o_q, o_sf, o_plain, flags, M)
    assert int(cnt.item()) == 5 + (o_cnt if with_cnt else 0)
    if clamp is not None:
        assert o_cnt > 0
    # the sentinel outside the written entries survives
    ref_free = oracle.sf_buffer(M, G, flags, ld)[0]
    written = np.ascontiguousarray(o_sf).view(np.uint8) != np.ascontiguousarray(ref_free).view(np.uint8)
    gpu_raw = np.ascontiguousarray(np_(sf)).view(np.uint8)
    if flags & ops.SF_UE8M0:
        assert (gpu_raw[~written] == 0xAB).all()
    else:
        w32 = written.reshape(-1, 4).any(axis=1)
        assert np.isnan(np_(sf).reshape(-1)[~w32]).all()


def test_swiglu_ex_without_count_or_options_matches_plain_entry():
    x = _swiglu_x(64, 512, seed=3).to(DEV)
    q0, sf0 = ops.swiglu_cast_fp8(x)
    q1, sf1 = ops.swiglu_cast_fp8_ex(x)
    assert torch.equal(q0, q1) and torch.equal(sf0, sf1)


def test_swiglu_ex_empty_rows():
    x = torch.empty(0, 512, dtype=torch.bfloat16, device=DEV)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    q, sf = ops.swiglu_cast_fp8_ex(x, clamp=1.0, clamp_count=cnt, sf_flags=7, sf_ld=0)
    assert q.shape == (0, 256) and int(cnt.item()) == 0


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
@pytest.mark.parametrize("clamp", [2.5, 2.51])
@pytest.mark.parametrize("count", [True, False])
def test_swiglu_clamp_fast_path_boundaries(fmt, clamp, count):
    """One value per row at, just above or just below c (2.51 is not a bf16
    value; 2.515625 is the next one above it), in the gate or as |up|, among
    values far below c.  Only values strictly above c are clamped and
    counted, wherever in the warp they sit (bf16 steps are 2^-6 near 2.5):
    with the count, through the warp-level skip test and the loop that
    clamps and counts; without it, through the clamp of every value."""
    M, N = 64, 256
    g = torch.Generator().manual_seed(11)
    x = (torch.rand(M, 2 * N, generator=g) - 0.5).to(torch.bfloat16)
    cases = [2.515625, 2.5, 2.484375, -2.515625]       # above / at / below 2.5, and a negative one
    expect = 0
    for r in range(M):
        v = cases[r % len(cases)]
        col = (r * 37) % N
        if r % 2 == 0:
            x[r, col] = v                                  # gate
            expect += v > clamp
        else:
            x[r, N + col] = v                              # up: |v| is compared
            expect += abs(v) > clamp
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    cnt_arg = cnt if count else None
    xb = oracle.bf16_bits(x)
    if fmt == "fp8":
        q, sf = ops.swiglu_cast_fp8_ex(x.to(DEV), clamp=clamp, clamp_count=cnt_arg)
        o_q, o_sf, o_cnt = oracle.swiglu_cast_fp8_ex(xb, clamp=clamp)
        check_swiglu_opts(np_(q), np_(sf), o_q, o_sf, o_sf, 0, M)
    else:
        q, sf = ops.swiglu_cast_fp4(x.to(DEV), group=32, clamp=clamp, clamp_count=cnt_arg)
        o_q, o_sf, o_cnt = oracle.swiglu_cast_fp4(xb, group=32, clamp=clamp)
        check_swiglu_opts(np_(q), np_(sf), o_q, o_sf, o_sf, 0, M, ordinal=fp4_ordinal)
    assert o_cnt == expect
    assert int(cnt.item()) == (expect if count else 0)


@pytest.mark.parametrize("fmt", ["fp8", "fp4"])
@pytest.mark.parametrize("count", [True, False])
def test_swiglu_variants_many_tiles_per_warp(fmt, count):
    """Enough rows (8191 x 2x2048) that the instances on a persistent grid
    (those with the clamp count) stride over five or six tiles per warp, with
    a ragged last stride, and the others take the grid of one tile per warp:
    clamp 7 on N(0, 2^2) values (about 0.07 % of the (gate, up) pairs exceed
    it, so about a third of the warp tiles clamp and count and the rest take
    the skip test's fast path), per-row weights, packed UE8M0 column-major
    scales.
    Every row against the oracle, and the count exact: each tile counted once."""
    M, N = 8191, 2048
    x = _swiglu_x(M, N, seed=17)
    w = torch.rand(M, generator=torch.Generator().manual_seed(18))
    flags = 7
    cnt = torch.full((1,), 3, dtype=torch.int64, device=DEV)
    xb = oracle.bf16_bits(x)
    if fmt == "fp8":
        G = N // 128
        sf, ld = _sentinel_sf(M, G, flags, (M + 3) // 4 * 4)
        q, _ = ops.swiglu_cast_fp8_ex(x.to(DEV), clamp=7.0, weights=w.to(DEV),
                                      clamp_count=cnt if count else None, sf_flags=flags,
                                      sf_ld=ld, out_sf=sf)
        o_q, o_sf, o_cnt = oracle.swiglu_cast_fp8_ex(xb, clamp=7.0, weights=w.numpy(),
                                                     flags=flags, ld=ld)
        _, o_plain, _ = oracle.swiglu_cast_fp8_ex(xb, clamp=7.0, weights=w.numpy())
        check_swiglu_opts(np_(q), np_(sf), o_q, o_sf, o_plain, flags, M)
    else:
        G = N // 32
        sf, ld = _sentinel_sf(M, G, flags, (M + 3) // 4 * 4)
        q, _ = ops.swiglu_cast_fp4(x.to(DEV), group=32, clamp=7.0, weights=w.to(DEV),
                                   clamp_count=cnt if count else None, sf_flags=flags,
                                   sf_ld=ld, out_sf=sf)
        o_q, o_sf, o_cnt = oracle.swiglu_cast_fp4(xb, group=32, clamp=7.0, weights=w.numpy(),
                                                  flags=flags, ld=ld)
        _, o_plain, _ = oracle.swiglu_cast_fp4(xb, group=32, clamp=7.0, weights=w.numpy())
        check_swiglu_opts(np_(q), np_(sf), o_q, o_sf, o_plain, flags, M, ordinal=fp4_ordinal)
    assert 1000 < o_cnt < 100000
    assert int(cnt.item()) == 3 + (o_cnt if count else 0)
    assert ops.device_status() == 0
