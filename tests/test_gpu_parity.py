"""GPU parity: every op through the C ABI against the CPU oracle.

Small ragged shapes compare every element here; the benchmarked sizes are
compared element by element in test_gpu_full_size.py.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops, workloads
from tests.parity_util import (assert_equal, assert_f32_bits_equal, assert_weights_close,
                               check_combine_bf16, check_combine_f32, check_swiglu)

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


def bits(t):
    return oracle.bf16_bits(t)


def np_(t):
    return t.detach().cpu().numpy()


# ---------------------------------------------------------------- top-k

TOPK_CASES = [(1, 16, 1), (31, 16, 2), (33, 32, 8), (64, 16, 2), (100, 64, 8), (257, 256, 8),
              (50, 384, 8), (40, 1024, 32), (10, 17, 17), (129, 100, 5), (8, 1, 1),
              (77, 8, 2), (45, 12, 3), (63, 16, 16), (3, 5, 5), (61, 512, 8), (37, 300, 6),
              (19, 384, 32), (23, 500, 20), (29, 512, 32)]


@pytest.mark.parametrize("T,E,k", TOPK_CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_topk_gate_parity(T, E, k, ties):
    inp = workloads.random_small(T, E, k, 128, seed=T * 7 + E + k, ties=ties)
    s = inp["scores"]
    idx, w = ops.topk_gate(s.to(DEV), k)
    o_idx, o_w = oracle.topk_gate(s.numpy(), k)
    assert_equal(np_(idx), o_idx, "topk_idx")
    assert_weights_close(np_(w), o_w)


TOPK_SWEEP_E = list(range(1, 41)) + [48, 63, 64, 65, 96, 127, 128, 129, 200, 255, 256, 257, 300,
                                     383, 384, 385, 448, 511, 512, 513, 700, 1024]


@pytest.mark.parametrize("E", TOPK_SWEEP_E)
def test_topk_gate_every_form_over_e(E):
    """Every top-k form (several tokens per warp for E <= 16, the rescan form
    for 16 < E <= 32 and E > 512, the candidate filter with 2 to 16 slots per
    lane in between, float4 rows where E is a multiple of 128) on seeded
    scores with forced ties, a random k and a token count that leaves the
    last warp's tokens partly empty."""
    rng = np.random.default_rng(E)
    k = int(rng.integers(1, min(E, 32) + 1))
    T = int(rng.integers(1, 200)) * 2 + 1
    inp = workloads.random_small(T, E, k, 128, seed=1000 + E, ties=bool(E % 2))
    s = inp["scores"]
    idx, w = ops.topk_gate(s.to(DEV), k)
    o_idx, o_w = oracle.topk_gate(s.numpy(), k)
    assert_equal(np_(idx), o_idx, f"topk_idx E={E} k={k}")
    assert_weights_close(np_(w), o_w, f"topk_w E={E} k={k}")


# (E, k) for every top-k form; T is 2.5 times the tokens one pass of the
# form's capped grid covers (1216 blocks: 32 tokens each for E <= 8, 16 for
# E <= 16, 8 otherwise), so each warp takes two or three tokens and the last
# pass is ragged
TOPK_STRIDE_CASES = [(8, 2), (16, 4), (32, 8), (64, 6), (128, 8), (200, 5), (256, 4),
                     (384, 8), (512, 8), (1024, 8)]


@pytest.mark.parametrize("E,k", TOPK_STRIDE_CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_topk_gate_grid_stride(E, k, ties):
    """Every top-k form with more tokens than its grid covers in one pass,
    random and heavily tied scores (the tied rows take the candidate filter's
    sorted-merge fallback where it has one)."""
    per_block = 32 if E <= 8 else 16 if E <= 16 else 8
    T = 1216 * per_block * 5 // 2 + 3
    inp = workloads.random_small(T, E, k, 128, seed=E * 31 + k, ties=ties)
    s = inp["scores"]
    idx, w = ops.topk_gate(s.to(DEV), k)
    o_idx, o_w = oracle.topk_gate(s.numpy(), k)
    assert_equal(np_(idx), o_idx, f"topk_idx E={E} k={k} T={T}")
    assert_weights_close(np_(w), o_w, f"topk_w E={E} k={k} T={T}")
    assert ops.device_status() == 0


@pytest.mark.parametrize("E", [8, 16, 384, 512])
def test_topk_gate_special_values_other_forms(E):
    """-0 and +0 tie (lower index first), +inf and -inf are ordinary values,
    and an all-equal row gives experts 0..k-1, in the several-tokens-per-warp
    form (E <= 16) and the forms for 256 < E <= 512."""
    row0 = [-0.0, 0.0, float("inf"), -float("inf"), float("inf"), -5.0] + [-7.0] * (E - 6)
    s = torch.tensor([row0, [1.0] * E, [-float("inf")] * E, row0[::-1]], dtype=torch.float32)
    idx, _ = ops.topk_gate(s.to(DEV), 6, weights=False)
    o_idx, _ = oracle.topk_gate(s.numpy(), 6, weights=False)
    assert_equal(np_(idx), o_idx, "topk_idx special")
    assert np_(idx)[1].tolist() == [0, 1, 2, 3, 4, 5]
    _, w = ops.topk_gate(s[1:2].to(DEV), 6)      # the finite row's weights
    assert np.allclose(np_(w), 1.0 / 6.0, rtol=4e-6, atol=0)


def test_topk_gate_special_values():
    s = torch.tensor([[-0.0, 0.0, float("inf"), -float("inf"), float("inf"), -5.0] + [-7.0] * 26,
                      [1.0] * 32, [-float("inf")] * 32], dtype=torch.float32)
    idx, _ = ops.topk_gate(s.to(DEV), 6, weights=False)
    o_idx, _ = oracle.topk_gate(s.numpy(), 6, weights=False)
    assert_equal(np_(idx), o_idx, "topk_idx special")
    assert np_(idx)[1].tolist() == [0, 1, 2, 3, 4, 5]


def test_topk_gate_empty():
    idx, w = ops.topk_gate(torch.empty(0, 16, device=DEV), 2)
    assert idx.shape == (0, 2)


# ---------------------------------------------------------------- route map

def _random_idx(T, E, k, seed, skew=False):
    g = torch.Generator().manual_seed(seed)
    if skew:
        base = torch.arange(k, dtype=torch.int32)
        return base.repeat(T, 1).contiguous()
    return torch.rand(T, E, generator=g).argsort(dim=1)[:, :k].to(torch.int32).contiguous()


@pytest.mark.parametrize("T,E,k", [(1, 16, 1), (127, 16, 2), (128, 16, 2), (129, 16, 2),
                                   (1000, 256, 8), (4133, 256, 8), (300, 1024, 32), (64, 1, 1),
                                   (513, 33, 3), (200003, 256, 8)])   # last: 391 chunks
def test_route_map_parity(T, E, k):
    idx = _random_idx(T, E, k, seed=T + E)
    out = ops.route_map(idx.to(DEV), E)
    ref = oracle.route_map(idx.numpy(), E)
    for name, a, b in zip(("counts", "offsets", "pos", "sorted_src"), out, ref):
        assert_equal(np_(a), b, name)


def test_route_map_skewed_and_deterministic():
    T, E, k = 3000, 256, 8
    idx = _random_idx(T, E, k, 0, skew=True).to(DEV)
    a = ops.route_map(idx, E)
    b = ops.route_map(idx, E)
    ref = oracle.route_map(np_(idx), E)
    for x, y, r in zip(a, b, ref):
        assert_equal(np_(x), r, "skewed route map")
        assert torch.equal(x, y)


def test_route_map_zero_tokens():
    counts, offsets, pos, src = ops.route_map(torch.empty(0, 2, dtype=torch.int32, device=DEV), 16)
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0


def test_route_map_flags_out_of_range_expert():
    idx = torch.tensor([[0, 1], [2, 16], [3, -1]], dtype=torch.int32, device=DEV)
    counts, offsets, pos, src = ops.route_map(idx, 16)
    assert ops.device_status() == ops.MOE_DEVERR_EXPERT_RANGE
    p = np_(pos)
    assert p[1, 1] == -1 and p[2, 1] == -1
    assert int(np_(counts).sum()) == 4
    assert sorted(p[p >= 0].tolist()) == [0, 1, 2, 3]


def test_route_map_flags_repeated_expert():
    idx = torch.tensor([[0, 1], [2, 2], [3, 4]], dtype=torch.int32, device=DEV)
    ops.route_map(idx, 8)
    assert ops.device_status() & ops.MOE_DEVERR_DUPLICATE_EXPERT


# ---------------------------------------------------------------- expand + cast

@pytest.mark.parametrize("T,H,k", [(1, 128, 1), (3, 384, 2), (33, 256, 8), (64, 256, 2),
                                   (200, 4096, 8), (37, 7168, 8), (5, 1152, 32),
                                   (4, 16384, 3), (3, 20480, 2)])   # largest row form; tile form
def test_expand_cast_parity(T, H, k):
    inp = workloads.random_small(T, 16, k, H, seed=T + H, zero_groups=True)
    x = inp["x"]
    pos = workloads.random_permutation_pos(T, k, seed=H)
    q, sf = ops.expand_cast_fp8(x.to(DEV), pos.to(DEV))
    o_q, o_sf = oracle.expand_cast_fp8(bits(x), pos.numpy())
    assert_equal(np_(q), o_q, "expand q")
    assert_f32_bits_equal(np_(sf), o_sf, "expand sf")


def test_expand_cast_extreme_values():
    H = 512
    rows = []
    bf = torch.finfo(torch.bfloat16)
    rows.append(torch.full((H,), bf.max))                       # saturating amax
    rows.append(torch.full((H,), -bf.tiny))                    # smallest normal, floor
    r = torch.zeros(H)
    r[::2] = -0.0
    rows.append(r)                                              # signed zeros
    r = torch.linspace(-3e4, 3e4, H)
    rows.append(r)
    r = torch.randn(H) * 1e-38                                  # subnormal bf16 values
    rows.append(r)
    r = torch.randn(H)
    r[7] = 1e30                                                 # one huge outlier
    rows.append(r)
    x = torch.stack(rows).to(torch.bfloat16)
    T = x.shape[0]
    pos = workloads.random_permutation_pos(T, 2, seed=1)
    q, sf = ops.expand_cast_fp8(x.to(DEV), pos.to(DEV))
    o_q, o_sf = oracle.expand_cast_fp8(bits(x), pos.numpy())
    assert_equal(np_(q), o_q, "extreme q")
    assert_f32_bits_equal(np_(sf), o_sf, "extreme sf")


@pytest.mark.parametrize("H", [256, 512])   # row form (H/128 = 2), bulk-store form (H/128 = 4)
def test_expand_dropped_copies_and_untouched_rows(H):
    T, k, R = 40, 4, 200
    x = workloads.random_small(T, 16, k, H, seed=3)["x"]
    g = torch.Generator().manual_seed(5)
    pos = torch.randperm(R, generator=g)[:T * k].to(torch.int32).view(T, k)
    pos[::3, 1] = -1                                            # dropped copies
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sf = torch.zeros(R, H // 128, device=DEV)
    ops.expand_cast_fp8(x.to(DEV), pos.to(DEV), R, out=q, out_sf=sf)
    o_q, o_sf = oracle.expand_cast_fp8(bits(x), pos.numpy(), num_rows=R, fill=0xAB)
    assert_equal(np_(q), o_q, "expand q with holes")
    assert_f32_bits_equal(np_(sf), o_sf, "expand sf with holes")


@pytest.mark.parametrize("H", [256, 512])
def test_expand_flags_pos_out_of_range(H):
    T, k = 4, 2
    x = workloads.random_small(T, 16, k, H, seed=4)["x"].to(DEV)
    pos = torch.tensor([[0, 1], [2, 3], [4, 8], [5, 6]], dtype=torch.int32, device=DEV)
    q = torch.zeros(8, H, dtype=torch.uint8, device=DEV)
    sf = torch.zeros(8, H // 128, device=DEV)
    ops.expand_cast_fp8(x, pos, 8, out=q, out_sf=sf)
    assert ops.device_status() == ops.MOE_DEVERR_POS_RANGE
    assert int(q[7].sum()) == 0


# ---------------------------------------------------------------- SwiGLU

@pytest.mark.parametrize("M,N,scale", [(1, 128, 1.0), (7, 256, 4.0), (100, 2048, 1.0),
                                       (1000, 384, 20.0), (33, 1024, 0.01)])
def test_swiglu_cast_parity(M, N, scale):
    g = torch.Generator().manual_seed(M + N)
    x = (torch.randn(M, 2 * N, generator=g) * scale).to(torch.bfloat16)
    q, sf = ops.swiglu_cast_fp8(x.to(DEV))
    o_q, o_sf = oracle.swiglu_cast_fp8(bits(x))
    check_swiglu(np_(q), np_(sf), o_q, o_sf)


def test_swiglu_cast_limits():
    N = 256
    gate = torch.tensor([0.0, 100.0, -120.0, -200.0, 3.0, -3.0] * 43)[:N]
    up = torch.tensor([3.0, 1.5, 5.0, -5.0, -0.0, 2.0] * 43)[:N]
    x = torch.cat([gate, up])[None, :].to(torch.bfloat16)
    q, sf = ops.swiglu_cast_fp8(x.to(DEV))
    o_q, o_sf = oracle.swiglu_cast_fp8(bits(x))
    check_swiglu(np_(q), np_(sf), o_q, o_sf)


# ---------------------------------------------------------------- combine

@pytest.mark.parametrize("T,H,k", [(1, 8, 1), (5, 256, 2), (64, 256, 2), (77, 4096, 8),
                                   (9, 7168, 8), (13, 512, 9), (4, 1024, 32), (7, 136, 3),
                                   (3, 20480, 2)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_combine_parity(T, H, k, dtype):
    g = torch.Generator().manual_seed(T * H + k)
    R = T * k + 3
    y = torch.randn(R, H, generator=g).to(torch.bfloat16)
    w = torch.rand(T, k, generator=g)
    pos = torch.randperm(R, generator=g)[:T * k].to(torch.int32).view(T, k)
    if k > 1:
        pos[::4, -1] = -1
    out = ops.combine(y.to(DEV), w.to(DEV), pos.to(DEV), dtype)
    o32, o16, mag = oracle.combine(bits(y), w.numpy(), pos.numpy())
    if dtype == torch.float32:
        check_combine_f32(np_(out), o32, mag)
    else:
        check_combine_bf16(bits(out.cpu()), o16, o32, mag)


def test_combine_one_hot_is_exact():
    T, k, H = 50, 8, 512
    g = torch.Generator().manual_seed(1)
    y = torch.randn(T * k, H, generator=g).to(torch.bfloat16)
    pos = workloads.random_permutation_pos(T, k, seed=2)
    w = torch.zeros(T, k)
    hot = torch.randint(0, k, (T,), generator=g)
    w[torch.arange(T), hot] = 1.0
    out = ops.combine(y.to(DEV), w.to(DEV), pos.to(DEV))
    assert torch.equal(out.cpu(), y[pos[torch.arange(T), hot].long()])


def test_combine_flags_pos_out_of_range():
    y = torch.ones(4, 256, dtype=torch.bfloat16, device=DEV)
    w = torch.ones(2, 2, device=DEV)
    pos = torch.tensor([[0, 1], [2, 4]], dtype=torch.int32, device=DEV)
    out = ops.combine(y, w, pos, torch.float32)
    assert ops.device_status() == ops.MOE_DEVERR_POS_RANGE
    assert torch.equal(out.cpu(), torch.tensor([[2.0] * 256, [1.0] * 256]))


# ---------------------------------------------------------------- streams, launches

def test_side_stream_and_launch_count():
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(w, device=DEV)
    ref_idx, _ = ops.topk_gate(inp["scores"], w.k)
    n0 = ops.launch_count()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        idx, _ = ops.topk_gate(inp["scores"], w.k)
    st.synchronize()
    assert ops.launch_count() == n0 + 1
    assert torch.equal(idx, ref_idx)


# ---------------------------------------------------------------- whole workloads

def _chain(w, inp):
    idx, wt = ops.topk_gate(inp["scores"], w.k)
    counts, offsets, pos, src = ops.route_map(idx, w.E)
    q, sf = ops.expand_cast_fp8(inp["x"], pos)
    out = {"idx": idx, "w": wt, "counts": counts, "offsets": offsets, "pos": pos, "src": src,
           "q": q, "sf": sf}
    if "y" in inp:
        out["comb16"] = ops.combine(inp["y"], wt, pos, torch.bfloat16)
        out["comb32"] = ops.combine(inp["y"], wt, pos, torch.float32)
    return out


def _route_oracle(w, inp):
    o_idx, o_w = oracle.topk_gate(np_(inp["scores"]), w.k)
    return (o_idx, o_w) + oracle.route_map(o_idx, w.E)


@pytest.mark.parametrize("name", ["tiny", "decode_1k"])
def test_small_workloads_every_element(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w, seed=0, device=DEV, with_y=True)
    got = _chain(w, inp)
    assert ops.device_status() == 0
    o_idx, o_w, o_counts, o_off, o_pos, o_src = _route_oracle(w, inp)
    assert_equal(np_(got["idx"]), o_idx, "idx")
    assert_weights_close(np_(got["w"]), o_w)
    for n, r in (("counts", o_counts), ("offsets", o_off), ("pos", o_pos), ("src", o_src)):
        assert_equal(np_(got[n]), r, n)
    o_q, o_sf = oracle.expand_cast_fp8(bits(inp["x"]), o_pos)
    assert_equal(np_(got["q"]), o_q, "q")
    assert_f32_bits_equal(np_(got["sf"]), o_sf, "sf")
    o32, o16, mag = oracle.combine(bits(inp["y"]), o_w, o_pos)
    check_combine_f32(np_(got["comb32"]), o32, mag)
    check_combine_bf16(bits(got["comb16"].cpu()), o16, o32, mag)


# ---------------------------------------------------------------- padded layout

@pytest.mark.parametrize("T,E,k,align", [(1000, 256, 8, 128), (37, 16, 2, 4), (513, 33, 3, 32),
                                         (300, 1024, 32, 64), (129, 16, 2, 1), (5, 64, 4, 256)])
def test_route_map_aligned_parity(T, E, k, align):
    idx = _random_idx(T, E, k, seed=T + E + align)
    got = ops.route_map_aligned(idx.to(DEV), E, align)
    ref = oracle.route_map_aligned(idx.numpy(), E, align)
    for name, a, b in zip(("counts", "offsets", "pos", "sorted_src"), got, ref):
        assert_equal(np_(a), b, name)
    assert ops.device_status() == 0


def test_route_map_aligned_flags_short_buffer():
    T, E, k, align = 64, 16, 2, 128
    idx = _random_idx(T, E, k, seed=3).to(DEV)
    counts, offsets, pos, src = ops.route_map_aligned(idx, E, align, num_rows=T * k)
    assert ops.device_status() & ops.MOE_DEVERR_ROWS_SHORT
    p = np_(pos)
    assert ((p == -1) | ((p >= 0) & (p < T * k))).all()


@pytest.mark.parametrize("T,E,k,H,align", [(200, 64, 8, 7168, 128), (37, 16, 2, 256, 16),
                                           (64, 8, 4, 512, 128), (33, 32, 3, 384, 8)])
def test_expand_padded_parity(T, E, k, H, align):
    inp = workloads.random_small(T, E, k, H, seed=T + H + align, zero_groups=True)
    x = inp["x"]
    idx = _random_idx(T, E, k, seed=T + align)
    _, _, o_pos, o_src = oracle.route_map_aligned(idx.numpy(), E, align)
    R = o_src.size
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sf = torch.full((R, H // 128), float("nan"), device=DEV)
    _, _, pos, src = ops.route_map_aligned(idx.to(DEV), E, align)
    ops.expand_cast_fp8_padded(x.to(DEV), pos, src, out=q, out_sf=sf)
    assert ops.device_status() == 0
    o_q, o_sf = oracle.expand_cast_fp8_padded(bits(x), o_pos, o_src)
    assert_equal(np_(q), o_q, "padded q")
    assert_f32_bits_equal(np_(sf), o_sf, "padded sf")


def test_expand_padded_no_tokens_zero_fills():
    H, R = 512, 100
    src = torch.full((R,), -1, dtype=torch.int32, device=DEV)
    q = torch.full((R, H), 0xAB, dtype=torch.uint8, device=DEV)
    sf = torch.full((R, H // 128), 7.0, device=DEV)
    ops.expand_cast_fp8_padded(torch.empty(0, H, dtype=torch.bfloat16, device=DEV),
                               torch.empty(0, 2, dtype=torch.int32, device=DEV), src,
                               out=q, out_sf=sf)
    assert int(q.abs().sum()) == 0 and float(sf.abs().sum()) == 0.0


def test_padded_chain_feeds_combine():
    # the padded pos works unchanged for combine (rows are looked up by pos)
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.make_inputs(w, seed=0, device=DEV)
    idx, wt = ops.topk_gate(inp["scores"], w.k)
    _, offsets, pos, src = ops.route_map_aligned(idx, w.E, 16)
    R = src.shape[0]
    g = torch.Generator().manual_seed(0)
    y = torch.randn(R, w.H, generator=g).to(torch.bfloat16)
    out = ops.combine(y.to(DEV), wt, pos, torch.float32)
    o32, _, mag = oracle.combine(bits(y), np_(wt), np_(pos))
    check_combine_f32(np_(out), o32, mag)
