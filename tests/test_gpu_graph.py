"""The decode-shaped call captured in a CUDA graph (as a serving loop would run
it): one capture of moe_route_expand_cast_fp8 with the library's own choice
of path, replayed on fresh inputs copied into the captured buffers, must give
the oracle's results every time.  Covers the one-launch replicated form, the
top-k + route/expand form, the separate launches, and the chained form."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops, workloads
from tests.parity_util import assert_equal, assert_f32_bits_equal, assert_weights_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
E, K, H = 256, 8, 1024


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


@pytest.mark.parametrize("T,mode", [(16, ops.PATH_AUTO), (200, ops.PATH_AUTO),
                                    (1500, ops.PATH_AUTO), (1500, ops.PATH_CHAINED)])
def test_captured_call_replays_on_new_inputs(T, mode):
    """AUTO: one launch / top-k + one / the separate launches; CHAINED: its
    three launches, including the scan's count of finished CTAs, which each
    replay must leave at zero for the next."""
    L = ops.lib()
    i32 = dict(dtype=torch.int32, device=DEV)
    scores = torch.empty(T, E, device=DEV)
    x = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    outs = [torch.empty(T, K, **i32), torch.empty(T, K, device=DEV), torch.empty(E, **i32),
            torch.empty(E + 1, **i32), torch.empty(T, K, **i32), torch.empty(T * K, **i32),
            torch.empty(T * K, H, dtype=torch.uint8, device=DEV),
            torch.empty(T * K, H // 128, device=DEV)]
    ws = ops.route_expand_cast_workspace(T, E, K, x)
    stream = torch.cuda.Stream(device=DEV)

    def call():
        rc = L.moe_route_expand_cast_fp8(scores.data_ptr(), T, E, K, x.data_ptr(), H,
                                         *[o.data_ptr() for o in outs], ws.data_ptr(), ws.numel(),
                                         mode, 128, ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0

    first = workloads.random_small(T, E, K, H, seed=T)
    scores.copy_(first["scores"])
    x.copy_(first["x"])
    with torch.cuda.stream(stream):
        call()                      # the first call outside the capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        call()
    for seed in (T + 1, T + 2, T + 3):
        inp = workloads.random_small(T, E, K, H, seed=seed, ties=seed % 2 == 0)
        scores.copy_(inp["scores"])
        x.copy_(inp["x"])
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert ops.device_status() == 0
        o_idx, o_w = oracle.topk_gate(inp["scores"].numpy(), K)
        o_c, o_o, o_p, o_s = oracle.route_map(o_idx, E)
        o_q, o_sf = oracle.expand_cast_fp8(oracle.bf16_bits(inp["x"]), o_p)
        for got, ref, name in ((outs[0], o_idx, "idx"), (outs[2], o_c, "counts"),
                               (outs[3], o_o, "offsets"), (outs[4], o_p, "pos"),
                               (outs[5], o_s, "sorted_src"), (outs[6], o_q, "q")):
            assert_equal(np_(got), ref, name)
        assert_weights_close(np_(outs[1]), o_w)
        assert_f32_bits_equal(np_(outs[7]), o_sf, "sf")
    del graph
