"""GPU parity of the chained route + expand (moe_route_expand_cast_fp8 with
MOE_PATH_CHAINED, a selectable form): the top-k kernel
that also ranks each copy within its chunk of tokens and counts the chunk's
copies, the column scan, and the expand that places its own copies.

Every output is compared with the oracle element by element (idx and the
route map bit-exact, weights within the top-k tolerance, codes and scale bits
bit-exact) on ragged shapes: T across the chunk sizes (16, 32 and 64 tokens)
and not a multiple of them, E not a multiple of 32, k from 1 to 32, ties; and
with the separate calls bit for bit.  Back-to-back calls on one workspace,
with different shapes, check that nothing a call leaves behind changes the
next call's result.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops, workloads
from tests.parity_util import assert_equal, assert_f32_bits_equal, assert_weights_close

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


def _check(scores, x, k, res):
    idx, w, counts, offsets, pos, src, q, sf = res
    E = scores.shape[1]
    o_idx, o_w = oracle.topk_gate(scores.numpy(), k)
    o_counts, o_off, o_pos, o_src = oracle.route_map(o_idx, E)
    o_q, o_sf = oracle.expand_cast_fp8(oracle.bf16_bits(x), o_pos)
    assert_equal(np_(idx), o_idx, "topk_idx")
    assert_weights_close(np_(w), o_w)
    for n, a, b in (("counts", counts, o_counts), ("offsets", offsets, o_off), ("pos", pos, o_pos),
                    ("sorted_src", src, o_src), ("q", q, o_q)):
        assert_equal(np_(a), b, n)
    assert_f32_bits_equal(np_(sf), o_sf, "sf")


CASES = [(1, 64, 2, 512), (15, 256, 8, 512), (16, 256, 8, 512), (17, 256, 8, 512),
         (100, 33, 32, 512), (1000, 100, 5, 1024), (1025, 256, 8, 7168), (4133, 256, 8, 512),
         (16384, 256, 8, 512), (16385, 256, 8, 512), (20001, 128, 6, 512), (32768, 64, 2, 512),
         (32769, 256, 8, 512), (40003, 200, 9, 512), (3000, 256, 1, 1024), (777, 160, 17, 2048)]


@pytest.mark.parametrize("T,E,k,H", CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_chained_matches_oracle(T, E, k, H, ties):
    inp = workloads.random_small(T, E, k, H, seed=T + E + k, ties=ties, zero_groups=True)
    s, x = inp["scores"], inp["x"]
    res = ops.route_expand_cast_fp8(s.to(DEV), x.to(DEV), k, mode=ops.PATH_CHAINED)
    assert ops.device_status() == 0
    _check(s, x, k, res)


@pytest.mark.parametrize("T,E,k,H", [(5000, 256, 8, 1536), (40000, 96, 4, 512)])
def test_chained_equals_separate_calls(T, E, k, H):
    inp = workloads.random_small(T, E, k, H, seed=T, ties=True)
    s, x = inp["scores"].to(DEV), inp["x"].to(DEV)
    a = ops.route_expand_cast_fp8(s, x, k, mode=ops.PATH_CHAINED)
    b = ops.route_expand_cast_fp8(s, x, k, mode=ops.PATH_SEPARATE)
    assert ops.device_status() == 0
    for i, (u, v) in enumerate(zip(a, b)):
        assert torch.equal(u.view(torch.uint8), v.view(torch.uint8)), f"output {i}"


def test_chained_back_to_back_on_one_workspace():
    """A second and third call on the same workspace, with other shapes,
    still match the oracle, and the control words stay zero."""
    T0, E, k = 20000, 256, 8
    ws = ops.route_expand_cast_workspace(T0, E, k, torch.empty(1, device=DEV))
    outs = []
    for T, H, seed in ((20000, 512, 1), (3000, 1024, 2), (17, 512, 3)):
        inp = workloads.random_small(T, E, k, H, seed=seed)
        res = ops.route_expand_cast_fp8(inp["scores"].to(DEV), inp["x"].to(DEV), k,
                                        mode=ops.PATH_CHAINED, workspace=ws)
        outs.append((inp["scores"], inp["x"], res))
    assert ops.device_status() == 0
    assert int(ws[:256].view(torch.int32).abs().sum()) == 0   # control words left at zero
    for s, x, res in outs:
        _check(s, x, k, res)


@pytest.mark.parametrize("E,k,H", [(32, 4, 512), (512, 8, 512), (256, 8, 384)])
def test_chained_refuses_shapes_it_does_not_handle(E, k, H):
    """E <= 32, E > 256 and H / 128 not a multiple of 4 are outside the chained
    form (AUTO takes the separate launches there)."""
    inp = workloads.random_small(2000, E, k, H, seed=E)
    s, x = inp["scores"].to(DEV), inp["x"].to(DEV)
    with pytest.raises(ops.MoeError) as ei:
        ops.route_expand_cast_fp8(s, x, k, mode=ops.PATH_CHAINED)
    assert ei.value.rc == ops.MOE_ERR_UNSUPPORTED
    res = ops.route_expand_cast_fp8(s, x, k, mode=ops.PATH_AUTO)
    assert ops.device_status() == 0
    _check(inp["scores"], inp["x"], k, res)
