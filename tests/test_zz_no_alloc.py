"""moe_route_map_noalloc: the route map for callers that cannot allocate.

Callers such as engine plugins, or runtimes that hand out every device buffer
from their own arena, may not call cudaMalloc while they run, so they cannot
supply moe_route_map's workspace.  moe_route_map_noalloc keeps that scratch in
a static device array instead.  This test calls it through the C ABI several
times in a row, on different problems in both orders of size (a call that
needs more histogram rows than the one before it, and fewer), and requires
bit-identical results to moe_route_map with a caller-provided workspace; one
problem is also checked against the CPU oracle, so the comparison does not
rest only on the kernels the two entry points share.  It checks that a
problem too large for the static array, or a misaligned pointer, is refused
before anything launches, and that bad expert ids are reported through the
device error word like moe_route_map reports them.

This file is named to be collected last, so that a run stopping at the
first failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCRATCH_BYTES = 1 << 20   # MOE_ROUTE_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def L():
    from moe_routing_precision_gb300 import _build
    _build.build()
    oracle.build()
    torch.cuda.set_device(0)
    assert ops.device_status() == 0
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


NAMES = ("counts", "offsets", "pos", "sorted_src")


def test_noalloc_matches_route_map_on_calls_in_a_row(L):
    problems = [(5000, 64, 6, 2, False),      # 40 histogram rows of 64
                (65536, 256, 8, 1, True),     # then a larger one: 128 rows of 256 (128 KiB)
                (20000, 128, 4, 4, False),    # then a smaller one again
                (300, 128, 4, 3, False)]      # decode-sized: the one-launch map, no scratch
    results = []
    for T, E, k, seed, skew in problems:
        idx = _idx(T, E, k, seed, skew)
        results.append((idx, E, _no_alloc(L, idx, E), _with_workspace(L, idx, E)))
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    for _, _, got, ref in results:
        for name, a, b in zip(NAMES, got, ref):
            assert torch.equal(a, b), name
    # the prefill-sized problem against the CPU oracle as well
    idx, E, got, _ = results[1]
    for name, a, b in zip(NAMES, got, oracle.route_map(idx.cpu().numpy(), E)):
        assert (a.cpu().numpy() == b).all(), f"{name} differs from the oracle"


def test_noalloc_reports_bad_expert_ids(L):
    # 1200 tokens: past the one-launch map, so the scratch-backed kernels run
    idx = torch.tensor([[0, 1], [2, 16], [3, 3]] * 400, dtype=torch.int32, device=DEV)
    got = _no_alloc(L, idx, 16)
    bits = ops.device_status()
    assert bits & ops.MOE_DEVERR_EXPERT_RANGE and bits & ops.MOE_DEVERR_DUPLICATE_EXPERT
    assert int(got[2][1, 1]) == -1                 # the out-of-range copy is not placed
    assert ops.device_status() == 0


def test_noalloc_refuses_problems_beyond_its_scratch(L):
    E, k = 256, 8
    T = (SCRATCH_BYTES // (E * 4) + 1) * 512   # one 512-token chunk more than fits
    assert L.moe_route_map_workspace_bytes(T, E, k) > SCRATCH_BYTES
    launches = L.moe_kernel_launch_count()
    p = ctypes.c_void_p(0x10000)
    rc = L.moe_route_map_noalloc(p, T, E, k, p, p, p, p, None)
    assert rc == 2                              # MOE_ERR_UNSUPPORTED, nothing launched
    assert L.moe_kernel_launch_count() == launches


def test_noalloc_refuses_misaligned_pointers(L):
    T, E, k = 1000, 64, 4
    launches = L.moe_kernel_launch_count()
    good, odd = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10002)
    for i in range(5):   # each of the five arrays misaligned in turn
        args = [good] * 5
        args[i] = odd
        rc = L.moe_route_map_noalloc(args[0], T, E, k, *args[1:], None)
        assert rc == 1                          # MOE_ERR_INVALID_ARG, nothing launched
    assert L.moe_kernel_launch_count() == launches
