"""GPU parity of the decode paths of moe_route_expand_cast_fp8 (top-k gate,
route map and expand + E4M3 cast in one launch: FUSED, one cooperative launch;
REPLICATED, one ordinary launch with the routing repeated per block) against
the oracle, their agreement with the separate launches, path selection, and
the fused path's bounded-wait failure path (a signal that is never sent; no
fault, no hang)."""
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
    ops.debug_set(ops.DEBUG_SKIP_ROUTE_SIGNAL, 0)
    ops.debug_set(ops.DEBUG_WAIT_TIMEOUT_NS, 1_000_000_000)
    assert ops.device_status() == 0


def np_(t):
    return t.detach().cpu().numpy()


def _inputs(T, E, k, H, seed, ties=False):
    inp = workloads.random_small(T, E, k, H, seed=seed, ties=ties, zero_groups=True)
    return inp["scores"], inp["x"]


def _check_against_oracle(scores, x, k, res):
    idx, w, counts, offsets, pos, src, q, sf = res
    E = scores.shape[1]
    o_idx, o_w = oracle.topk_gate(scores.numpy(), k)
    o_counts, o_off, o_pos, o_src = oracle.route_map(o_idx, E)
    o_q, o_sf = oracle.expand_cast_fp8(oracle.bf16_bits(x), o_pos)
    assert_equal(np_(idx), o_idx, "topk_idx")
    assert_weights_close(np_(w), o_w)
    assert_equal(np_(counts), o_counts, "counts")
    assert_equal(np_(offsets), o_off, "offsets")
    assert_equal(np_(pos), o_pos, "pos")
    assert_equal(np_(src), o_src, "sorted_src")
    assert_equal(np_(q), o_q, "q")
    assert_f32_bits_equal(np_(sf), o_sf, "sf")


CASES = [(1, 64, 2, 128), (7, 256, 8, 4096), (100, 256, 8, 7168), (1024, 256, 8, 4096),
         (33, 128, 4, 384), (300, 64, 6, 1024), (2048, 256, 8, 512), (50, 256, 16, 256),
         (151, 96, 3, 640), (153, 256, 8, 16384)]


@pytest.mark.parametrize("T,E,k,H", CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_fused_matches_oracle(T, E, k, H, ties):
    scores, x = _inputs(T, E, k, H, seed=T + E + H, ties=ties)
    ws = ops.route_expand_cast_workspace(T, E, k, x.to(DEV))
    res = ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k, mode=ops.PATH_FUSED,
                                    workspace=ws)
    assert ops.device_status() == 0
    _check_against_oracle(scores, x, k, res)
    assert int(ws[:8].abs().sum()) == 0            # control words left zero


@pytest.mark.parametrize("T,E,k,H", [(64, 256, 8, 4096), (1000, 128, 4, 1024)])
def test_fused_equals_separate_launches(T, E, k, H):
    scores, x = _inputs(T, E, k, H, seed=5)
    s, xd = scores.to(DEV), x.to(DEV)
    a = ops.route_expand_cast_fp8(s, xd, k, mode=ops.PATH_FUSED)
    b = ops.route_expand_cast_fp8(s, xd, k, mode=ops.PATH_SEPARATE)
    assert ops.device_status() == 0
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.uint8) if u.dtype == torch.float32 else u,
                           v.view(torch.uint8) if v.dtype == torch.float32 else v)


def test_back_to_back_calls_share_a_workspace():
    T, E, k, H = 256, 256, 8, 2048
    ws = ops.route_expand_cast_workspace(T, E, k, torch.empty(1, device=DEV))
    outs = []
    for seed in range(4):                           # no synchronisation between the calls
        scores, x = _inputs(T, E, k, H, seed=seed)
        outs.append((scores, x, ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k,
                                                          mode=ops.PATH_FUSED, workspace=ws)))
    assert ops.device_status() == 0
    for scores, x, res in outs:
        _check_against_oracle(scores, x, k, res)


def test_path_launch_counts_and_auto_choice():
    E, k, H = 256, 8, 512
    for T, mode, launches in [(512, ops.PATH_FUSED, 1), (512, ops.PATH_REPLICATED, 2),
                              (32, ops.PATH_REPLICATED, 1), (33, ops.PATH_REPLICATED, 2),
                              (4096, ops.PATH_AUTO, 4), (32, ops.PATH_AUTO, 1),
                              (512, ops.PATH_AUTO, 2), (1024, ops.PATH_AUTO, 2),
                              (1025, ops.PATH_AUTO, 4), (1024, ops.PATH_SEPARATE, 3),
                              (1025, ops.PATH_SEPARATE, 4), (512, ops.PATH_CHAINED, 3)]:
        scores, x = _inputs(T, E, k, H, seed=T)
        s, xd = scores.to(DEV), x.to(DEV)
        ws = ops.route_expand_cast_workspace(T, E, k, xd)
        torch.cuda.synchronize()
        n0 = ops.launch_count()
        res = ops.route_expand_cast_fp8(s, xd, k, mode=mode, workspace=ws)
        assert ops.launch_count() - n0 == launches
        assert ops.device_status() == 0
        if T <= 1025:
            _check_against_oracle(scores, x, k, res)


@pytest.mark.parametrize("E,k", [(16, 2), (512, 8)])
def test_fused_refuses_shapes_it_does_not_handle(E, k):
    scores, x = _inputs(8, E, k, 256, seed=1)
    with pytest.raises(ops.MoeError) as ei:
        ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k, mode=ops.PATH_FUSED)
    assert ei.value.rc == ops.MOE_ERR_UNSUPPORTED
    res = ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k, mode=ops.PATH_AUTO)
    assert ops.device_status() == 0
    _check_against_oracle(scores, x, k, res)


def test_wait_that_runs_out_reports_timeout_and_leaves_a_usable_context():
    """Block 0 routes but never signals: every block's bounded wait runs out
    after 20 ms, the kernel sets MOE_DEVERR_TIMEOUT and finishes, and the
    control words are reset by the last block."""
    T, E, k, H = 200, 256, 8, 1024
    scores, x = _inputs(T, E, k, H, seed=3)
    s, xd = scores.to(DEV), x.to(DEV)
    ws = ops.route_expand_cast_workspace(T, E, k, xd)
    ops.debug_set(ops.DEBUG_WAIT_TIMEOUT_NS, 20_000_000)
    ops.debug_set(ops.DEBUG_SKIP_ROUTE_SIGNAL, 1)
    try:
        ops.route_expand_cast_fp8(s, xd, k, mode=ops.PATH_FUSED, workspace=ws)
        bits = ops.device_status()
    finally:
        ops.debug_set(ops.DEBUG_SKIP_ROUTE_SIGNAL, 0)
        ops.debug_set(ops.DEBUG_WAIT_TIMEOUT_NS, 1_000_000_000)
    assert bits == ops.MOE_DEVERR_TIMEOUT
    assert int(ws[:8].abs().sum()) == 0
    res = ops.route_expand_cast_fp8(s, xd, k, mode=ops.PATH_FUSED, workspace=ws)
    assert ops.device_status() == 0
    _check_against_oracle(scores, x, k, res)


@pytest.mark.parametrize("mode", [ops.PATH_AUTO, ops.PATH_FUSED, ops.PATH_SEPARATE,
                                  ops.PATH_REPLICATED, ops.PATH_CHAINED])
def test_no_tokens(mode):
    E, k, H = 64, 4, 256
    s = torch.empty(0, E, device=DEV)
    x = torch.empty(0, H, dtype=torch.bfloat16, device=DEV)
    res = ops.route_expand_cast_fp8(s, x, k, mode=mode)
    assert ops.device_status() == 0
    assert int(res[2].abs().sum()) == 0 and int(res[3].abs().sum()) == 0   # counts, offsets
    assert res[6].shape == (0, H)


# ---------------------------------------------------------------- replicated path

# T <= 32: one launch (selection repeated per block); above: top-k launch + route/expand
REP_CASES = [(1, 64, 2, 128), (7, 256, 8, 4096), (100, 256, 8, 7168), (33, 128, 4, 384),
             (300, 64, 6, 1024), (512, 256, 8, 512), (128, 256, 32, 256), (151, 96, 3, 640),
             (153, 256, 8, 8192), (16, 200, 1, 128), (64, 33, 32, 256), (40, 256, 9, 2048),
             (32, 256, 8, 1024), (33, 256, 8, 1024), (1024, 256, 8, 4096), (2048, 256, 8, 512),
             (700, 256, 23, 256), (500, 40, 5, 128), (500, 33, 32, 256)]


@pytest.mark.parametrize("T,E,k,H", REP_CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_replicated_matches_oracle(T, E, k, H, ties):
    scores, x = _inputs(T, E, k, H, seed=T + 3 * E + H, ties=ties)
    res = ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k, mode=ops.PATH_REPLICATED)
    assert ops.device_status() == 0
    _check_against_oracle(scores, x, k, res)


@pytest.mark.parametrize("T,E,k,H", [(64, 256, 8, 4096), (200, 128, 4, 1024)])
def test_replicated_equals_separate_launches(T, E, k, H):
    scores, x = _inputs(T, E, k, H, seed=6)
    s, xd = scores.to(DEV), x.to(DEV)
    a = ops.route_expand_cast_fp8(s, xd, k, mode=ops.PATH_REPLICATED)
    b = ops.route_expand_cast_fp8(s, xd, k, mode=ops.PATH_SEPARATE)
    assert ops.device_status() == 0
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.uint8) if u.dtype == torch.float32 else u,
                           v.view(torch.uint8) if v.dtype == torch.float32 else v)


def test_replicated_back_to_back_calls():
    T, E, k, H = 96, 256, 8, 2048
    outs = []
    for seed in range(4):                           # no synchronisation between the calls
        scores, x = _inputs(T, E, k, H, seed=20 + seed)
        outs.append((scores, x, ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k,
                                                          mode=ops.PATH_REPLICATED)))
    assert ops.device_status() == 0
    for scores, x, res in outs:
        _check_against_oracle(scores, x, k, res)


@pytest.mark.parametrize("T,E,k,H", [(2049, 256, 8, 256), (1100, 256, 16, 256), (8, 16, 2, 256),
                                     (8, 512, 8, 256), (8, 256, 8, 8320), (300, 256, 8, 8320)])
def test_replicated_refuses_shapes_it_does_not_handle(T, E, k, H):
    scores, x = _inputs(T, E, k, H, seed=2)
    with pytest.raises(ops.MoeError) as ei:
        ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k, mode=ops.PATH_REPLICATED)
    assert ei.value.rc == ops.MOE_ERR_UNSUPPORTED
    res = ops.route_expand_cast_fp8(scores.to(DEV), x.to(DEV), k, mode=ops.PATH_AUTO)
    assert ops.device_status() == 0
    _check_against_oracle(scores, x, k, res)

