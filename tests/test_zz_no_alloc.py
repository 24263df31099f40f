"""moe_route_map_noalloc: the route map for callers that cannot allocate.

Callers such as engine plugins, or runtimes that hand out every device buffer
from their own arena, may not call cudaMalloc while they run, so they cannot
supply moe_route_map's workspace.  moe_route_map_noalloc keeps that scratch in
a static device array instead.  This test calls it through the C ABI twice in
a row, on different problems (so a second call that leaned on the first
call's leftovers would show), and requires bit-identical results to
moe_route_map with a caller-provided workspace.  It also checks that a
problem too large for the static array is refused before anything launches.

This file is named to be collected last, so that a run stopping at the
first failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH_BYTES = 1 << 20   # MOE_ROUTE_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def L():
    from moe_routing_precision_gb300 import _build, ops
    _build.build()
    torch.cuda.set_device(0)
    return ops.lib()


def _outputs(T, E, k):
    i32 = dict(dtype=torch.int32, device=DEV)
    # filled with garbage so nothing passes by accident
    return [torch.full((E,), -7, **i32), torch.full((E + 1,), -7, **i32),
            torch.full((T, k), -7, **i32), torch.full((T * k,), -7, **i32)]


def _idx(T, E, k, seed, skew):
    g = torch.Generator().manual_seed(seed)
    if skew:   # every token on the same few experts: long runs, empty experts
        base = torch.randperm(E, generator=g)[:k].to(torch.int32)
        return base.repeat(T, 1).contiguous().to(DEV)
    return torch.rand(T, E, generator=g).argsort(1)[:, :k].to(torch.int32).contiguous().to(DEV)


def _with_workspace(L, idx, E):
    T, k = idx.shape
    outs = _outputs(T, E, k)
    ws = torch.empty(L.moe_route_map_workspace_bytes(T, E, k), dtype=torch.uint8, device=DEV)
    s = torch.cuda.current_stream().cuda_stream or None
    rc = L.moe_route_map(idx.data_ptr(), T, E, k, *[o.data_ptr() for o in outs], ws.data_ptr(),
                         ws.numel(), s)
    assert rc == 0
    return outs


def _no_alloc(L, idx, E):
    T, k = idx.shape
    outs = _outputs(T, E, k)
    s = torch.cuda.current_stream().cuda_stream or None
    rc = L.moe_route_map_noalloc(idx.data_ptr(), T, E, k, *[o.data_ptr() for o in outs], s)
    assert rc == 0
    return outs


def test_noalloc_matches_route_map_on_two_calls_in_a_row(L):
    problems = [(65536, 256, 8, 1, True),     # prefill-sized, skewed (512 KiB of scratch)
                (5000, 64, 6, 2, False),      # a smaller problem right after it
                (300, 128, 4, 3, False)]      # decode-sized: the one-launch map, no scratch
    results = []
    for T, E, k, seed, skew in problems:
        idx = _idx(T, E, k, seed, skew)
        results.append((_no_alloc(L, idx, E), _with_workspace(L, idx, E)))
    torch.cuda.synchronize()
    for got, ref in results:
        for name, a, b in zip(("counts", "offsets", "pos", "sorted_src"), got, ref):
            assert torch.equal(a, b), name


def test_noalloc_refuses_problems_beyond_its_scratch(L):
    E, k = 256, 8
    T = (SCRATCH_BYTES // (E * 4) + 1) * 512   # one 512-token chunk more than fits
    assert L.moe_route_map_workspace_bytes(T, E, k) > SCRATCH_BYTES
    launches = L.moe_kernel_launch_count()
    rc = L.moe_route_map_noalloc(ctypes.c_void_p(0x10000), T, E, k, ctypes.c_void_p(0x10000),
                                 ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10000),
                                 ctypes.c_void_p(0x10000), None)
    assert rc == 2                              # MOE_ERR_UNSUPPORTED, nothing launched
    assert L.moe_kernel_launch_count() == launches
