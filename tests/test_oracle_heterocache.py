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


# ------------------------------------------------ Phase 1: medians over steps
def test_stability_hand_worked():
    """Prefill set {1,2,3,4}; decoding sets {1,2,3,4} (overlap 1), {1,2,9,10}
    (1/2), {7,8,9,10} (0): the median of (1, 1/2, 0) is 1/2.  A fourth step
    {1,2,3,9} (3/4) makes T even: the median is (1/2 + 3/4) / 2 = 5/8."""
    pre = [[1, 2, 3, 4]]
    dec = [[[1, 2, 3, 4]], [[1, 2, 9, 10]], [[7, 8, 9, 10]]]
    per, st = Hc.stability_over_steps(dec, pre)
    assert per[:, 0].tolist() == [1.0, 0.5, 0.0] and st.tolist() == [0.5]
    per, st = Hc.stability_over_steps(dec + [[[1, 2, 3, 9]]], pre)
    assert per[:, 0].tolist() == [1.0, 0.5, 0.0, 0.75] and st.tolist() == [0.625]


def test_similarity_hand_worked():
    """Two steps, three heads.  Step 0: A={1,2,3,4}, B={1,2,5,6}, C={7,8}:
    maxima (1/2, 1/2, 0).  Step 1: A={1,2,3,4}, B={1,2,3,4}, C={4,9}:
    maxima (1, 1, 1/2).  Medians of two values: (3/4, 3/4, 1/4)."""
    steps = [[[1, 2, 3, 4], [1, 2, 5, 6], [7, 8]], [[1, 2, 3, 4], [1, 2, 3, 4], [4, 9]]]
    per, sim = Hc.similarity_over_steps(steps)
    assert per.tolist() == [[0.5, 0.5, 0.0], [1.0, 1.0, 0.5]]
    assert sim.tolist() == [0.75, 0.75, 0.25]


def test_median_against_exact_brute_force():
    """statistics.median over exact rationals of the fp32 values, rounded once."""
    from fractions import Fraction
    import statistics
    rng = np.random.default_rng(5)
    for T in (1, 2, 7, 100, 101):
        x = (rng.integers(0, 64, (T, 5)) / np.float32(rng.integers(1, 64))).astype(np.float32)
        want = [np.float32(float(statistics.median([Fraction(float(v)) for v in x[:, h]]))) for h in range(5)]
        assert Hc.median_over_steps(x).tolist() == [float(w) for w in want]
        # the median is not the mean, and is taken over steps, not heads
        assert Hc.median_over_steps(np.array([[0.0], [0.0], [1.0]], dtype=np.float32)).tolist() == [0.0]


def _median_mean(x):
    return np.asarray(x, dtype=np.float32).astype(np.float64).mean(axis=0).astype(np.float32)


def _median_max(x):
    return np.asarray(x, dtype=np.float32).max(axis=0)


def _median_lower_middle(x):
    v = np.sort(np.asarray(x, dtype=np.float32), axis=0)
    return v[(v.shape[0] - 1) // 2]


def _median_over_heads(x):
    x = np.asarray(x, dtype=np.float32)
    return np.full(x.shape[1], np.median(x[0]), dtype=np.float32)


@pytest.mark.parametrize("mutant", [_median_mean, _median_max, _median_lower_middle, _median_over_heads])
def test_median_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(Hc, "median_over_steps", mutant)
    failed = 0
    for pin in (test_stability_hand_worked, test_similarity_hand_worked, test_median_against_exact_brute_force):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0
