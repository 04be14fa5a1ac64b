"""Pins of the oracle's top-k selection against an independent statement of
it: an entry is among the k largest of its row iff fewer than k entries rank
above it, where an entry ranks above another when its value is larger, or
equal at a smaller index; the result lists them by that rank."""
import numpy as np
import pytest

import oracle


def brute_topk(row: np.ndarray, k: int):
    n = len(row)
    rank = [sum(1 for i in range(n) if row[i] > row[j] or (row[i] == row[j] and i < j))
            for j in range(n)]
    ids = sorted((j for j in range(n) if rank[j] < k), key=lambda j: rank[j])
    return np.array(ids), row[ids]


def test_hand_example():
    L = np.array([[3.0, 1.0, 3.0, 2.0, -5.0]])
    ids, vals = oracle.topk(L, 3)
    assert ids.tolist() == [[0, 2, 3]]
    assert vals.tolist() == [[3.0, 3.0, 2.0]]
    ids, _ = oracle.topk(L, 5)
    assert ids.tolist() == [[0, 2, 3, 1, 4]]


@pytest.mark.parametrize("seed", range(6))
def test_against_rank_definition(seed):
    rng = np.random.default_rng(seed)
    M, N = 5, 23
    L = rng.integers(-3, 4, size=(M, N)).astype(np.float64)  # many ties
    L[0] = 0.0
    L[1, 7] = -0.0
    for k in (1, 2, 7, N):
        ids, vals = oracle.topk(L, k)
        for m in range(M):
            bi, bv = brute_topk(L[m], k)
            assert ids[m].tolist() == bi.tolist()
            assert np.array_equal(vals[m], bv)


def test_distinct_values_match_a_full_sort():
    rng = np.random.default_rng(9)
    L = rng.standard_normal((3, 1000))
    ids, vals = oracle.topk(L, 50)
    for m in range(3):
        assert np.array_equal(vals[m], np.sort(L[m])[::-1][:50])
        assert np.array_equal(L[m, ids[m]], vals[m])
