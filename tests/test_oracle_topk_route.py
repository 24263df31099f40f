"""Pins of the oracle's top-k gate, top-k weights and route map.

Top-k (TileKernels page, 2.1): brute force over all k-subsets on tiny inputs,
forced ties, k = E, +-inf, torch.topk on distinct scores.  Weights: sum to 1,
torch.softmax in float64 over the selected scores, the closed-form ratio
w_i / w_j = exp(s_i - s_j).  Route map ("CuTeDSL at Perplexity", local
dispatch): invariants, and numpy's stable argsort as an independent routine.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle


def _brute_topk(row, k):
    """Best k-subset by exhaustive search: maximise the sorted score vector,
    then prefer the lexicographically smaller index tuple, which is what
    'ties go to the lower index' means for a set; then order it."""
    E = len(row)
    best = None
    for sub in itertools.combinations(range(E), k):
        key = (sorted((row[i] for i in sub), reverse=True), [-i for i in sub])
        if best is None or key > best[0]:
            best = (key, sub)
    sub = best[1]
    return sorted(sub, key=lambda i: (-row[i], i))


@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    T, E, k = 12, 7, 3
    scores = rng.integers(-2, 3, size=(T, E)).astype(np.float32)  # many ties
    idx, _ = oracle.topk_gate(scores, k, weights=False)
    for t in range(T):
        assert list(idx[t]) == _brute_topk(list(scores[t]), k)


def test_topk_all_equal_rows_and_k_equals_E():
    s = np.zeros((3, 16), np.float32)
    idx, w = oracle.topk_gate(s, 5)
    assert (idx == np.arange(5)).all()
    assert np.allclose(w, 0.2, rtol=0, atol=1e-7)
    rng = np.random.default_rng(3)
    s = rng.standard_normal((5, 9)).astype(np.float32)
    idx, _ = oracle.topk_gate(s, 9, weights=False)
    for t in range(5):
        assert sorted(idx[t]) == list(range(9))
        assert list(idx[t]) == list(np.argsort(-s[t], kind="stable"))


def test_topk_duplicate_maximum_picks_lower_index():
    s = np.array([[0.5, 2.0, -1.0, 2.0, 2.0, 1.0]], np.float32)
    idx, _ = oracle.topk_gate(s, 4, weights=False)
    assert list(idx[0]) == [1, 3, 4, 5]


def test_topk_signed_zero_ties_and_infinities():
    s = np.array([[-0.0, 0.0, np.inf, -np.inf, np.inf, -5.0]], np.float32)
    idx, _ = oracle.topk_gate(s, 6, weights=False)
    # +inf (2, 4), then the two zeros in index order (-0 == +0), -5, -inf
    assert list(idx[0]) == [2, 4, 0, 1, 5, 3]


def test_topk_nan_rejected():
    s = np.array([[0.0, np.nan, 1.0]], np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.topk_gate(s, 1)


def test_topk_matches_torch_topk_on_distinct_scores():
    g = torch.Generator().manual_seed(4)
    s = torch.randn(200, 256, generator=g)
    vals, ref = torch.topk(s, 8, dim=1, largest=True, sorted=True)
    idx, _ = oracle.topk_gate(s.numpy(), 8, weights=False)
    assert np.array_equal(idx, ref.numpy().astype(np.int32))


def test_weights_softmax_over_selected():
    g = torch.Generator().manual_seed(5)
    s = torch.randn(300, 64, generator=g) * 3
    idx, w = oracle.topk_gate(s.numpy(), 6)
    sel = torch.gather(s.double(), 1, torch.from_numpy(idx).long())
    ref = torch.softmax(sel, dim=1).float().numpy()
    assert np.allclose(w, ref, rtol=2e-7, atol=0)
    assert np.allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
    # ratio closed form
    r = w[:, 1].astype(np.float64) / w[:, 0]
    e = np.exp(sel[:, 1].numpy() - sel[:, 0].numpy())
    assert np.allclose(r, e, rtol=1e-6)
    # weights follow the score order
    assert (np.diff(w, axis=1) <= 0).all()


def test_weights_k1_is_one():
    s = np.random.default_rng(6).standard_normal((10, 32)).astype(np.float32)
    _, w = oracle.topk_gate(s, 1)
    assert (w == 1.0).all()


# ---------------------------------------------------------------- route map

def _check_route_invariants(idx, E, counts, offsets, pos, src):
    T, k = idx.shape
    R = T * k
    assert counts.sum() == R and offsets[0] == 0 and offsets[E] == R
    assert (np.diff(offsets) == counts).all()
    assert np.array_equal(np.sort(pos.ravel()), np.arange(R))          # bijection
    assert np.array_equal(src[pos.ravel()], np.arange(R))               # inverse
    assert np.array_equal(pos.ravel()[src], np.arange(R))
    flat = idx.ravel()
    for e in range(E):
        seg = src[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg // k) > 0).all()                             # stable by token


@pytest.mark.parametrize("T,E,k,seed", [(1, 4, 1, 0), (37, 16, 2, 1), (100, 64, 8, 2),
                                        (513, 256, 8, 3), (64, 9, 9, 4)])
def test_route_map_invariants_and_stable_argsort(T, E, k, seed):
    rng = np.random.default_rng(seed)
    s = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = oracle.topk_gate(s, k, weights=False)
    counts, offsets, pos, src = oracle.route_map(idx, E)
    _check_route_invariants(idx, E, counts, offsets, pos, src)
    # an independent routine: numpy's stable sort of the flattened expert ids
    ref_src = np.argsort(idx.ravel(), kind="stable").astype(np.int32)
    assert np.array_equal(src, ref_src)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E).astype(np.int32))


def test_route_map_worked_example():
    # 3 tokens, E=4, k=2 (worked by hand from the definition)
    idx = np.array([[2, 0], [0, 3], [2, 3]], np.int32)
    counts, offsets, pos, src = oracle.route_map(idx, 4)
    assert list(counts) == [2, 0, 2, 2]
    assert list(offsets) == [0, 2, 2, 4, 6]
    # expert 0: (0,1),(1,0) -> rows 0,1; expert 2: (0,0),(2,0) -> 2,3;
    # expert 3: (1,1),(2,1) -> 4,5
    assert pos.tolist() == [[2, 0], [1, 4], [3, 5]]
    assert list(src) == [1, 2, 0, 4, 3, 5]


def test_route_map_skewed_and_empty_experts():
    idx = np.tile(np.array([[5, 1]], np.int32), (50, 1))
    counts, offsets, pos, src = oracle.route_map(idx, 8)
    _check_route_invariants(idx, 8, counts, offsets, pos, src)
    assert counts[1] == 50 and counts[5] == 50 and counts.sum() == 100


def test_route_map_rejects_out_of_range_index():
    with pytest.raises(oracle.OracleError):
        oracle.route_map(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(oracle.OracleError):
        oracle.route_map(np.array([[-1, 2]], np.int32), 4)


def test_route_map_empty():
    counts, offsets, pos, src = oracle.route_map(np.zeros((0, 3), np.int32), 5)
    assert (counts == 0).all() and (offsets == 0).all() and pos.size == 0 and src.size == 0
