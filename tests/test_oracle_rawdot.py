"""Pins of the INT8 raw inner-product scorer's oracle (CPU only).

Against a hand-worked example, the existing softmax oracle (its logits, and
its selection for a single query, where HillInfer's monotonicity argument
makes the rankings equal), and the analytic rounding bound.
"""

import json
import os

import numpy as np
import pytest

from oracle import kvc_oracle as O
from oracle import rawdot_int8 as R


def test_hand_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "int8_hand_example.json")))
    codes, scale = R.quantize_int8(np.array(g["x"], dtype=np.float32))
    assert codes.tolist() == g["codes"]
    assert scale == np.float32(np.float32(g["scale_num"]) / np.float32(g["scale_den"]))
    qb = R.summed_query(np.array(g["q_rows"], dtype=np.float32))
    qc, _ = R.quantize_int8(qb)
    assert qc.tolist() == g["q_codes"]
    assert int(np.dot(qc, codes)) == g["dot"]
    s = R.raw_scores_int8(np.array(g["q_rows"], dtype=np.float32), np.array([g["x"]], dtype=np.float32))
    assert s[0] == np.float32(np.float32(np.float32(g["dot"]) * scale) * scale)


def test_codes_span_and_zero_rows():
    rng = np.random.default_rng(3)
    for _ in range(50):
        x = rng.standard_normal(64).astype(np.float32) * rng.uniform(0.01, 50)
        c, s = R.quantize_int8(x)
        assert np.abs(c).max() == 127
        assert c[np.argmax(np.abs(x))] == np.sign(x[np.argmax(np.abs(x))]) * 127
        assert np.all(np.abs(x - c * np.float64(s)) <= 0.5 * np.float64(s) * (1 + 1e-6))
    c, s = R.quantize_int8(np.zeros(16, dtype=np.float32))
    assert not c.any() and s == 0
    assert R.raw_scores_int8(np.ones((2, 16), np.float32), np.zeros((3, 16), np.float32)).tolist() == [0, 0, 0]


@pytest.mark.parametrize("seed,G,W,S,D", [(0, 1, 1, 40, 8), (1, 2, 4, 64, 16), (2, 4, 8, 100, 32)])
def test_summed_query_is_the_softmax_free_window_group_sum(seed, G, W, S, D):
    # keys before the window are seen by every window query, so there the
    # sum of the oracle's logits times sqrt(D) is q_bar . k_j
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((G * W, D)).astype(np.float32)
    k = rng.standard_normal((S, D)).astype(np.float32)
    L = O.dense_logits(q.astype(np.float64), k.astype(np.float64), W)
    outside = np.arange(S) <= S - W
    ref = L[:, outside].sum(axis=0) * np.sqrt(D)
    np.testing.assert_allclose(R.raw_scores_exact(q, k)[outside], ref, rtol=1e-12, atol=1e-9)
    np.testing.assert_allclose(R.summed_query(q), q.astype(np.float64).sum(axis=0), rtol=1e-6, atol=1e-5)


@pytest.mark.parametrize("seed,scale", [(0, 1.0), (1, 0.01), (2, 30.0)])
def test_int8_scores_within_the_rounding_bound(seed, scale):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((8, 32)) * scale).astype(np.float32)
    k = (rng.standard_normal((200, 32)) * scale).astype(np.float32)
    k[7] = 0.0
    exact = k.astype(np.float64) @ R.summed_query(q).astype(np.float64)
    err = np.abs(R.raw_scores_int8(q, k).astype(np.float64) - exact)
    assert np.all(err <= R.int8_error_bound(q, k))
    # and the bound is not vacuous: it is far below the score spread
    assert np.median(R.int8_error_bound(q, k)) < 0.1 * np.std(exact)


@pytest.mark.parametrize("seed", range(4))
def test_single_query_raw_ranking_equals_softmax_selection(seed):
    # HillInfer, "Algorithmic Simplification": for one query the softmax is
    # monotone in q.k, so ranking by the raw product keeps the same keys
    rng = np.random.default_rng(seed)
    S, D, K_l, sink, recent = 80, 16, 20, 2, 1
    q = rng.standard_normal((1, D))
    k = rng.standard_normal((S, D))
    a = O.score_head(q, k, 1, 1)
    soft = O.select_topk(a["s"], K_l, sink, recent)
    raw = O.select_topk(R.raw_scores_exact(q, k), K_l, sink, recent)
    assert soft.tolist() == raw.tolist()


def test_selection_handles_negative_scores():
    s = np.array([-3.0, -1.0, -2.0, 5.0, -1.0, 0.0, -7.0, -1.0])
    idx = O.select_topk(s, 4, 1, 1)      # R = {0, 7}; best others: 3 (5.0), 5 (0.0)
    assert idx.tolist() == [0, 3, 5, 7]
    idx = O.select_topk(s, 5, 1, 1)      # ... then the tie at -1.0 goes to index 1
    assert idx.tolist() == [0, 1, 3, 5, 7]


def test_row_batched_scores_equal_the_per_key_ones():
    rng = np.random.default_rng(9)
    q = (rng.standard_normal((6, 64)) * 2).astype(np.float32)
    k = (rng.standard_normal((300, 64)) * rng.uniform(0.001, 100, (300, 1))).astype(np.float32)
    k[11] = 0.0
    a = R.raw_scores_int8(q, k)
    b = R.raw_scores_int8_rows(q, k)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_round_half_to_even_hand_case(golden_dir):
    # a row whose amax is 127 maps every element to itself, so each
    # fractional .5 is an exact tie; the codes were worked out by hand
    g = json.load(open(os.path.join(golden_dir, "int8_rounding_ties.json")))
    codes, scale = R.quantize_int8(np.array(g["x"], dtype=np.float32))
    assert codes.tolist() == g["codes"]
    assert scale == np.float32(g["scale"])
