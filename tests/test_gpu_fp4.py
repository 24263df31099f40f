"""GPU parity of the FP4 E2M1 expand + cast (TileKernels article, sections
3.1, 3.2 and 2.2 with the float4_e2m1fn output type) against the oracle:
packed codes and every scale-buffer byte bit-exact, for every group size,
scale layout, padded rows and the values at the edges of the format."""
import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops, workloads
from tests.parity_util import assert_equal, check_swiglu_opts, fp4_ordinal

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


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


def _raw_equal(gpu_sf, ref_sf, what):
    assert_equal(np.ascontiguousarray(np_(gpu_sf)).view(np.uint8),
                 np.ascontiguousarray(ref_sf).view(np.uint8), what)


def _sentinel_sf(rows, G, flags, ld):
    ref, ld = oracle.sf_buffer(rows, G, flags, ld)
    return torch.from_numpy(ref.copy()).to(DEV), ld


SHAPES = [(9, 256, 2), (13, 384, 3), (40, 512, 4), (21, 7168, 8), (5, 4096, 2), (3, 16384, 2)]


@pytest.mark.parametrize("group", [16, 32, 64, 128])
@pytest.mark.parametrize("flags", [0, 2, 6])
@pytest.mark.parametrize("T,H,k", SHAPES)
def test_expand_fp4_parity(group, flags, T, H, k):
    if H % group:
        pytest.skip("H not a multiple of the group")
    x = workloads.random_small(T, 16, k, H, seed=T * H + group + flags, zero_groups=True)["x"]
    R = T * k + 5                                   # rows no pos names stay untouched
    g = torch.Generator().manual_seed(group + H)
    pos = torch.randperm(R, generator=g)[:T * k].to(torch.int32).view(T, k)
    pos[::4, 0] = -1                                # dropped copies
    q = torch.full((R, H // 2), 0xAB, dtype=torch.uint8, device=DEV)
    sf, ld = _sentinel_sf(R, H // group, flags, None)
    ops.expand_cast_fp4(x.to(DEV), pos.to(DEV), R, group=group, sf_flags=flags, out=q, out_sf=sf)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp4(oracle.bf16_bits(x), pos.numpy(), num_rows=R, group=group,
                                       flags=flags)
    assert_equal(np_(q), o_q, f"fp4 q group={group} flags={flags}")
    _raw_equal(sf, o_sf, f"fp4 sf group={group} flags={flags}")


@pytest.mark.parametrize("flags,off", [(6, 1), (6, 4), (6, 8), (2, 4), (2, 16)])
@pytest.mark.parametrize("group,T,H,k", [(32, 21, 7168, 8), (16, 6, 7168, 20), (32, 9, 384, 5),
                                         (128, 11, 512, 32), (64, 3, 16384, 2)])
def test_expand_fp4_rowmajor_scales_at_offsets(flags, off, group, T, H, k):
    """Row-major scales (power-of-two f32, packed UE8M0 bytes) written into a
    buffer `off` bytes into an allocation: the byte rows go out 8, 4 or 1
    bytes per store, the f32 rows by bulk copy or per group; rows of 4 to 448
    entries, k up to 32.  The bytes around the buffer keep their fill."""
    x = workloads.random_small(T, 16, k, H, seed=T * H + off + group, zero_groups=True)["x"]
    R = T * k + 3
    g = torch.Generator().manual_seed(off + H + k + group)
    pos = torch.randperm(R, generator=g)[:T * k].to(torch.int32).view(T, k)
    pos[1::3, k - 1] = -1
    ref, _ = oracle.sf_buffer(R, H // group, flags)
    raw = np.ascontiguousarray(ref).view(np.uint8).reshape(-1)
    buf = torch.full((raw.size + off + 32,), 0x5C, dtype=torch.uint8, device=DEV)
    buf[off:off + raw.size] = torch.from_numpy(raw.copy()).to(DEV)
    q = torch.full((R, H // 2), 0xAB, dtype=torch.uint8, device=DEV)
    ops.expand_cast_fp4(x.to(DEV), pos.to(DEV), R, group=group, sf_flags=flags, out=q,
                        out_sf=buf[off:off + raw.size])
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp4(oracle.bf16_bits(x), pos.numpy(), num_rows=R, group=group,
                                       flags=flags)
    assert_equal(np_(q), o_q, "fp4 rowmajor q")
    got = np_(buf)
    assert_equal(got[off:off + raw.size], np.ascontiguousarray(o_sf).view(np.uint8).reshape(-1),
                 "fp4 rowmajor sf")
    assert (got[:off] == 0x5C).all() and (got[off + raw.size:] == 0x5C).all()


@pytest.mark.parametrize("group", [16, 32, 128])
@pytest.mark.parametrize("flags,staged", [(1, False), (1, True), (3, True), (7, False), (7, True)])
def test_expand_fp4_colmajor_and_padded(group, flags, staged):
    T, E, k, H, align = 60, 16, 4, 1024, 32
    x = workloads.random_small(T, E, k, H, seed=group + flags, zero_groups=True)["x"]
    g = torch.Generator().manual_seed(7)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    _, _, o_pos, o_src = oracle.route_map_aligned(idx.numpy(), E, align)
    R = o_src.size
    ld = (R + 3) // 4 * 4 + 4
    q = torch.full((R, H // 2), 0xAB, dtype=torch.uint8, device=DEV)
    sf, ld = _sentinel_sf(R, H // group, flags, ld)
    ops.expand_cast_fp4(x.to(DEV), torch.from_numpy(o_pos).to(DEV), group=group,
                        sorted_src=torch.from_numpy(o_src).to(DEV), sf_flags=flags, sf_ld=ld,
                        out=q, out_sf=sf, workspace=True if staged else None)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp4(oracle.bf16_bits(x), o_pos, sorted_src=o_src, group=group,
                                       flags=flags, ld=ld)
    assert_equal(np_(q), o_q, "fp4 padded q")
    _raw_equal(sf, o_sf, "fp4 padded sf")


@pytest.mark.parametrize("group", [16, 32])
def test_expand_fp4_format_edges(group):
    H = 512
    bf = torch.finfo(torch.bfloat16)
    rows = [torch.full((H,), bf.max), torch.full((H,), -bf.tiny), torch.zeros(H),
            torch.linspace(-3e4, 3e4, H), torch.randn(H) * 1e-38]
    r = torch.zeros(H)
    r[::2] = -0.0
    rows.append(r)
    r = torch.randn(H)
    r[5] = 1e30
    rows.append(r)
    # every E2M1 midpoint and value, times a group max of 6 (scale exactly 1)
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                         -0.25, -5.0])
    r = mids.repeat(H // 16)
    rows.append(r)
    r = torch.zeros(H)                              # multiply-by-inverse case
    r[0::group] = 0.030517578125
    r[1::group] = 0.003814697265625
    rows.append(r)
    x = torch.stack(rows).to(torch.bfloat16)
    T = x.shape[0]
    pos = workloads.random_permutation_pos(T, 2, seed=2)
    q, sf = ops.expand_cast_fp4(x.to(DEV), pos.to(DEV), group=group)
    o_q, o_sf = oracle.expand_cast_fp4(oracle.bf16_bits(x), pos.numpy(), group=group)
    assert_equal(np_(q), o_q, "fp4 edges q")
    _raw_equal(sf, o_sf, "fp4 edges sf")


def test_expand_fp4_flags_pos_out_of_range():
    T, k, H = 4, 2, 256
    x = workloads.random_small(T, 16, k, H, seed=4)["x"].to(DEV)
    pos = torch.tensor([[0, 1], [2, 3], [4, 8], [5, 6]], dtype=torch.int32, device=DEV)
    q = torch.zeros(8, H // 2, dtype=torch.uint8, device=DEV)
    sf = torch.zeros(8, H // 32, device=DEV)
    ops.expand_cast_fp4(x, pos, 8, group=32, out=q, out_sf=sf)
    assert ops.device_status() == ops.MOE_DEVERR_POS_RANGE
    assert int(q[7].sum()) == 0


@pytest.mark.parametrize("name", ["skewed_8k", "prefill_64k"])
def test_expand_fp4_full_size_every_row(name):
    """The skewed and prefill inputs, group 32 (the bench's FP4 launch): every
    copy of every token against the oracle's cast of that token (on token
    shards over the host's threads), compared on the device."""
    from tests import oracle_pool
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, seed=0, device=DEV)
    idx, _ = ops.topk_gate(inp["scores"], w.k)
    _, _, pos, _ = ops.route_map(idx, w.E)
    q, sf = ops.expand_cast_fp4(inp["x"], pos, group=32)
    assert ops.device_status() == 0
    o_q, o_sf = oracle_pool.per_token_cast_fp4(oracle.bf16_bits(inp["x"]), 32)
    o_q, o_sf = torch.from_numpy(o_q).to(DEV), torch.from_numpy(o_sf.view(np.int32)).to(DEV)
    sf_bits = sf.view(torch.int32)
    for j in range(w.k):
        rows = pos[:, j].long()
        assert torch.equal(q[rows], o_q), f"codes of copy {j}"
        assert torch.equal(sf_bits[rows], o_sf), f"scales of copy {j}"
    del inp, q, sf, o_q, o_sf
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- SwiGLU -> FP4

# (clamp, per-row weights, clamp count)
FP4_VARIANTS = {"plain": (None, False, False), "weight": (None, True, False),
                "clamp": (1.0, False, False), "clamp_count": (1.0, False, True),
                "clamp_weight_count": (1.0, True, True)}


@pytest.mark.parametrize("group", [16, 32, 64, 128])
@pytest.mark.parametrize("flags", [0, 1, 2, 7])
@pytest.mark.parametrize("variant", list(FP4_VARIANTS))
@pytest.mark.parametrize("M,N", [(1, 128), (7, 384), (100, 2048), (1000, 256)])
def test_swiglu_fp4_parity(group, flags, variant, M, N):
    if N % group:
        pytest.skip("N not a multiple of the group")
    g = torch.Generator().manual_seed(M + N + group + flags)
    x = (torch.randn(M, 2 * N, generator=g) * 2.0).to(torch.bfloat16)
    clamp, with_w, with_cnt = FP4_VARIANTS[variant]
    w = torch.rand(M, generator=g) if with_w else None
    ld = (M + 3) // 4 * 4 + 8 if flags & ops.SF_COLMAJOR else None
    sf, ld = _sentinel_sf(M, N // group, flags, ld)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    q, _ = ops.swiglu_cast_fp4(x.to(DEV), group=group, clamp=clamp,
                               weights=None if w is None else w.to(DEV),
                               clamp_count=cnt if with_cnt else None,
                               sf_flags=flags, sf_ld=ld, out_sf=sf)
    xb = oracle.bf16_bits(x)
    wn = None if w is None else w.numpy()
    o_q, o_sf, o_cnt = oracle.swiglu_cast_fp4(xb, group=group, clamp=clamp, weights=wn,
                                              flags=flags, ld=ld)
    _, o_plain, _ = oracle.swiglu_cast_fp4(xb, group=group, clamp=clamp, weights=wn)
    check_swiglu_opts(np_(q), np_(sf), o_q, o_sf, o_plain, flags, M, ordinal=fp4_ordinal)
    assert int(cnt.item()) == (o_cnt if with_cnt else 0)
    assert ops.device_status() == 0


def test_swiglu_fp4_full_size_every_row():
    """swiglu_64k (65536 rows x 2x2048), group 32: every row."""
    from tests import oracle_pool
    w = workloads.WORKLOADS["swiglu_64k"]
    hx = workloads.make_inputs(w, seed=0, device=DEV)["swiglu_x"]
    q, sf = ops.swiglu_cast_fp4(hx, group=32)
    assert ops.device_status() == 0
    o_q, o_sf = oracle_pool.swiglu_cast_fp4(oracle.bf16_bits(hx), 32)
    check_swiglu_opts(np_(q), np_(sf), o_q, o_sf, o_sf, 0, w.M, ordinal=fp4_ordinal)
    del hx, q, sf
    torch.cuda.empty_cache()


def test_fp4_empty_inputs_and_zero_fill_only():
    H, R = 512, 40
    src = torch.full((R,), -1, dtype=torch.int32, device=DEV)
    q = torch.full((R, H // 2), 0xAB, dtype=torch.uint8, device=DEV)
    sf = torch.full((R, H // 32), 7.0, device=DEV)
    ops.expand_cast_fp4(torch.empty(0, H, dtype=torch.bfloat16, device=DEV),
                        torch.empty(0, 2, dtype=torch.int32, device=DEV), group=32,
                        sorted_src=src, out=q, out_sf=sf)
    assert ops.device_status() == 0
    assert int(q.sum()) == 0 and float(sf.abs().sum()) == 0.0
    q2, sf2 = ops.swiglu_cast_fp4(torch.empty(0, 2 * H, dtype=torch.bfloat16, device=DEV), group=32)
    assert q2.shape == (0, H // 2) and sf2.shape == (0, H // 32)
