"""Pins of the HeteroCache overlap oracle (CPU only): closed forms of the
overlap coefficient, its symmetry and range, a hand-worked example, and the
similarity score as the row maximum of the pairwise matrix."""

import numpy as np
import pytest

from oracle import heterocache as Hc


def test_closed_forms():
    a = np.arange(10, 50)
    assert Hc.overlap_coefficient(a, a) == 1.0                       # identical
    assert Hc.overlap_coefficient(a, a + 100) == 0.0                 # disjoint
    assert Hc.overlap_coefficient(a[5:15], a) == 1.0                 # nested: min is the subset
    assert Hc.overlap_coefficient([], a) == 0.0                      # empty


def test_hand_example():
    # A = {1, 3, 5, 7}, B = {3, 4, 5}: |A n B| = 2, min(4, 3) = 3 -> 2/3
    assert Hc.overlap_coefficient([1, 3, 5, 7], [3, 4, 5]) == np.float32(2) / np.float32(3)


def test_symmetry_and_range():
    rng = np.random.default_rng(0)
    for _ in range(100):
        a = rng.choice(500, rng.integers(1, 200), replace=False)
        b = rng.choice(500, rng.integers(1, 200), replace=False)
        x = Hc.overlap_coefficient(a, b)
        assert x == Hc.overlap_coefficient(b, a)
        assert 0.0 <= x <= 1.0
        # against the plain count over a dense membership vector
        ma = np.zeros(500, bool); ma[a] = True
        mb = np.zeros(500, bool); mb[b] = True
        assert x == np.float32(np.float32((ma & mb).sum()) / np.float32(min(len(a), len(b))))


def test_similarity_is_the_row_max_of_the_pair_matrix():
    rng = np.random.default_rng(1)
    sets = [np.sort(rng.choice(300, 60, replace=False)) for _ in range(6)]
    sets[4] = sets[1][:30]            # a nested pair: both reach 1
    M = np.array([[Hc.overlap_coefficient(x, y) for y in sets] for x in sets])
    np.fill_diagonal(M, 0)
    sim = Hc.head_similarity(sets)
    assert np.array_equal(sim, M.max(axis=1).astype(np.float32))
    assert sim[1] == 1.0 and sim[4] == 1.0
    assert Hc.head_similarity([sets[0]]).tolist() == [0.0]
