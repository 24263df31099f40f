"""The sharded oracle runs (tests/oracle_pool.py) equal the whole-array oracle.

The full-size GPU parity tests compare against the oracle run on token or row
shards over host threads; these CPU tests check, on inputs a few shards
long, that the shards' concatenation is exactly the single-call result, with
the shard edges inside the arrays (several threads) and with one thread.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_routing_precision_gb300 import workloads
from tests import oracle_pool


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_sharded_topk_and_casts_equal_single_call(threads):
    T, E, k, H = 301, 64, 6, 512
    inp = workloads.random_small(T, E, k, H, seed=threads, ties=True, zero_groups=True)
    s = inp["scores"].numpy()
    xb = oracle.bf16_bits(inp["x"])
    i1, w1 = oracle.topk_gate(s, k)
    i2, w2 = oracle_pool.topk_gate(s, k, threads=threads)
    assert np.array_equal(i1, i2) and np.array_equal(w1.view(np.uint32), w2.view(np.uint32))
    q1, sf1 = oracle.per_token_cast(xb)
    q2, sf2 = oracle_pool.per_token_cast(xb, threads=threads)
    assert np.array_equal(q1, q2) and np.array_equal(sf1.view(np.uint32), sf2.view(np.uint32))
    ident = np.arange(T, dtype=np.int32)[:, None]
    for group in (16, 32):
        q1, sf1 = oracle.expand_cast_fp4(xb, ident, group=group)
        q2, sf2 = oracle_pool.per_token_cast_fp4(xb, group, threads=threads)
        assert np.array_equal(q1, q2) and np.array_equal(sf1.view(np.uint32), sf2.view(np.uint32))


@pytest.mark.parametrize("threads", [1, 5])
def test_sharded_swiglu_equals_single_call(threads):
    g = torch.Generator().manual_seed(threads)
    xb = oracle.bf16_bits((torch.randn(257, 2 * 256, generator=g) * 3).to(torch.bfloat16))
    q1, sf1 = oracle.swiglu_cast_fp8(xb)
    q2, sf2 = oracle_pool.swiglu_cast_fp8(xb, threads=threads)
    assert np.array_equal(q1, q2) and np.array_equal(sf1.view(np.uint32), sf2.view(np.uint32))
    q1, sf1, _ = oracle.swiglu_cast_fp4(xb, group=32)
    q2, sf2 = oracle_pool.swiglu_cast_fp4(xb, 32, threads=threads)
    assert np.array_equal(q1, q2) and np.array_equal(sf1.view(np.uint32), sf2.view(np.uint32))


@pytest.mark.parametrize("threads", [1, 4])
def test_sharded_combine_of_gathered_rows_equals_combine(threads):
    T, k, H = 97, 3, 136
    g = torch.Generator().manual_seed(threads)
    R = T * k + 5
    yb = oracle.bf16_bits(torch.randn(R, H, generator=g).to(torch.bfloat16))
    w = torch.rand(T, k, generator=g).numpy()
    pos = torch.randperm(R, generator=g)[:T * k].to(torch.int32).view(T, k).numpy()
    o32, o16, mag = oracle.combine(yb, w, pos)
    g32, g16, gmag = oracle_pool.combine_gathered(np.ascontiguousarray(yb[pos.reshape(-1)]), w,
                                                  threads=threads)
    assert np.array_equal(o32.view(np.uint32), g32.view(np.uint32))
    assert np.array_equal(o16, g16) and np.array_equal(mag, gmag)


def test_shard_bounds_cover_exactly():
    for n, parts in ((0, 4), (1, 4), (7, 3), (100, 7), (65536, 64)):
        b = oracle_pool.shard_bounds(n, parts)
        covered = [i for a, c in b for i in range(a, c)]
        assert covered == list(range(n))
