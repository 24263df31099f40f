"""Pins of the oracle's padded expert layout (route map with aligned
segments, expand with zero-filled padding rows).

align = 1 reduces to the plain route map (itself pinned against numpy's
stable argsort); for any align the segments are the plain route map's shifted
to aligned starts, padding rows are -1 and all-zero, and a hand-worked case
fixes the arithmetic.
"""
import numpy as np
import pytest

import oracle


def _idx(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)


def test_align_one_is_the_plain_route_map():
    idx = _idx(300, 64, 6, 0)
    c1, o1, p1, s1 = oracle.route_map(idx, 64)
    c2, o2, p2, s2 = oracle.route_map_aligned(idx, 64, 1)
    assert np.array_equal(c1, c2) and np.array_equal(o1, o2) and np.array_equal(p1, p2)
    assert np.array_equal(s1, s2[:300 * 6]) and s2.size == 300 * 6


@pytest.mark.parametrize("align,T,E,k,seed", [(128, 1000, 64, 8, 1), (4, 37, 16, 2, 2),
                                              (32, 513, 33, 3, 3), (128, 1, 8, 1, 4)])
def test_segments_are_aligned_shifts_of_the_plain_map(align, T, E, k, seed):
    idx = _idx(T, E, k, seed)
    c, o, p, s = oracle.route_map(idx, E)
    ca, oa, pa, sa = oracle.route_map_aligned(idx, E, align)
    assert np.array_equal(ca, c)
    assert (oa % align == 0).all() and oa[0] == 0
    assert np.array_equal(np.diff(oa), -(-c // align) * align)
    # each copy keeps its rank inside its expert's segment
    e = idx
    assert np.array_equal(pa - oa[e], p - o[e])
    real = np.zeros(sa.size, bool)
    real[pa.ravel()] = True
    assert (sa[~real] == -1).all()
    assert np.array_equal(sa[pa.ravel()], np.arange(T * k))
    assert sa.size == T * k + E * (align - 1)


def test_worked_example():
    # 3 tokens, E=3, k=2, align=4: counts [2,1,3] -> padded [4,4,4],
    # offsets [0,4,8,12]; expert 0 gets (0,1),(1,0); expert 1 gets (2,1);
    # expert 2 gets (0,0),(1,1),(2,0)
    idx = np.array([[2, 0], [0, 2], [2, 1]], np.int32)
    c, o, p, s = oracle.route_map_aligned(idx, 3, 4, num_rows=12)
    assert list(c) == [2, 1, 3]
    assert list(o) == [0, 4, 8, 12]
    assert p.tolist() == [[8, 0], [1, 9], [10, 4]]
    assert list(s) == [1, 2, -1, -1, 5, -1, -1, -1, 0, 3, 4, -1]


def test_too_few_rows_rejected():
    idx = _idx(10, 8, 2, 5)
    with pytest.raises(oracle.OracleError):
        oracle.route_map_aligned(idx, 8, 128, num_rows=100)


def test_padded_expand_zero_fills_exactly_the_padding_rows():
    rng = np.random.default_rng(6)
    T, E, k, H, align = 40, 8, 2, 256, 16
    idx = _idx(T, E, k, 7)
    import torch
    x = oracle.bf16_bits(torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16))
    _, _, pos, src = oracle.route_map_aligned(idx, E, align)
    q, sf = oracle.expand_cast_fp8_padded(x, pos, src)
    qt, sft = oracle.per_token_cast(x)
    pad = src < 0
    assert (q[pad] == 0).all() and (sf[pad] == 0).all()
    for t in range(T):
        for j in range(k):
            assert np.array_equal(q[pos[t, j]], qt[t]) and np.array_equal(sf[pos[t, j]], sft[t])
    assert not np.isnan(sf).any() and not (q == 0xAB).all(axis=1).any()
