"""GPU parity at the benchmarked sizes: every element of every output.

The skewed-routing workload (T=8192), the large prefill (T=65536) and the
SwiGLU workload (65536 rows of 2x2048) run through the C ABI, both as the
individual calls (the launches the bench times) and as the chained one-call
form, and every output element is compared with
the oracle: the whole top-k and route map, the E4M3 codes and scale bits of
all k copies of every token (bit-exact), combine for every token in both
output dtypes, and every SwiGLU row.  The oracle runs on token shards over
the host's threads (tests/oracle_pool.py), which gives exactly its
whole-array result.

Where the comparison is made on the device (the codes and scales of the k
copies: 3.8 GB at prefill size), the oracle's per-token result is copied to
the GPU and each copy j is gathered through pos[:, j]; a mismatch is located
and reported on the host.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import ops, workloads
from tests import oracle_pool
from tests.parity_util import (assert_equal, assert_weights_close, check_combine_bf16,
                               check_combine_f32, check_swiglu)

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


def _assert_rows_equal_on_device(got, ref_dev, what):
    """got, ref_dev: same-shape device tensors; report the first mismatch."""
    if torch.equal(got, ref_dev):
        return
    bad = (got != ref_dev).nonzero()
    i = tuple(int(v) for v in bad[0])
    raise AssertionError(f"{what}: {bad.shape[0]} elements differ; first at {i}: "
                         f"gpu={got[i].item()!r} oracle={ref_dev[i].item()!r}")


@pytest.mark.parametrize("path", ["calls", "chained"])
@pytest.mark.parametrize("name", ["skewed_8k", "prefill_64k"])
def test_full_size_every_element(name, path):
    """path "calls": moe_topk_gate, moe_route_map, moe_expand_cast_fp8 (the
    launches the bench times: its one-call AUTO path takes them at these
    sizes); "chained": moe_route_expand_cast_fp8 with MOE_PATH_CHAINED."""
    w = workloads.WORKLOADS[name]
    T, E, k, H, R, G = w.T, w.E, w.k, w.H, w.R, w.G
    inp = workloads.make_inputs(w, seed=0, device=DEV, with_y=True)
    if path == "calls":
        idx, wt = ops.topk_gate(inp["scores"], k)
        counts, offsets, pos, src = ops.route_map(idx, E)
        q, sf = ops.expand_cast_fp8(inp["x"], pos)
    else:
        n0 = ops.launch_count()
        idx, wt, counts, offsets, pos, src, q, sf = ops.route_expand_cast_fp8(
            inp["scores"], inp["x"], k, mode=ops.PATH_CHAINED)
        assert ops.launch_count() - n0 == 3          # the chained launches
    comb16 = ops.combine(inp["y"], wt, pos, torch.bfloat16)
    comb32 = ops.combine(inp["y"], wt, pos, torch.float32)
    assert ops.device_status() == 0

    # top-k and route map: whole arrays
    o_idx, o_w = oracle_pool.topk_gate(np_(inp["scores"]), k)
    assert_equal(np_(idx), o_idx, "topk_idx")
    assert_weights_close(np_(wt), o_w)
    o_counts, o_off, o_pos, o_src = oracle.route_map(o_idx, E)
    for n, a, r in (("counts", counts, o_counts), ("offsets", offsets, o_off), ("pos", pos, o_pos),
                    ("sorted_src", src, o_src)):
        assert_equal(np_(a), r, n)

    # expand + cast: every code and scale bit of all k copies of every token
    o_q, o_sf = oracle_pool.per_token_cast(oracle.bf16_bits(inp["x"]))
    o_q_dev = torch.from_numpy(o_q).to(DEV)
    o_sf_dev = torch.from_numpy(o_sf.view(np.int32)).to(DEV)
    del o_q, o_sf
    sf_bits = sf.view(torch.int32)
    for j in range(k):
        rows = pos[:, j].long()
        _assert_rows_equal_on_device(q[rows], o_q_dev, f"q copy {j}")
        _assert_rows_equal_on_device(sf_bits[rows], o_sf_dev, f"sf copy {j}")
    # every row of the output is some copy's (pos is a bijection onto [0, R))
    assert int(torch.bincount(pos.flatten().long(), minlength=R).min()) == 1
    del o_q_dev, o_sf_dev, q, sf
    torch.cuda.empty_cache()

    # combine, every token, in shards (the oracle gets each token's k rows)
    shard = 4096
    for a in range(0, T, shard):
        b = min(T, a + shard)
        rows = pos[a:b].flatten().long()
        ys = oracle.bf16_bits(inp["y"][rows])
        o32, o16, mag = oracle_pool.combine_gathered(ys, o_w[a:b])
        check_combine_f32(np_(comb32[a:b]), o32, mag)
        check_combine_bf16(oracle.bf16_bits(comb16[a:b]), o16, o32, mag)
    del inp, comb16, comb32
    torch.cuda.empty_cache()


def test_swiglu_workload_every_row():
    w = workloads.WORKLOADS["swiglu_64k"]
    x = workloads.make_inputs(w, seed=0, device=DEV)["swiglu_x"]
    q, sf = ops.swiglu_cast_fp8(x)
    assert ops.device_status() == 0
    o_q, o_sf = oracle_pool.swiglu_cast_fp8(oracle.bf16_bits(x))
    frac = check_swiglu(np_(q), np_(sf), o_q, o_sf)
    assert frac <= 1e-3
    del x, q, sf
    torch.cuda.empty_cache()
