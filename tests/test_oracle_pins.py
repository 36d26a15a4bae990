"""Pins of the fp64 oracle against things other than itself (CPU only).

Each check ties the oracle to a brute force, a hand-worked example, a closed
form, a library routine in a special case, or an invariant the pages state
(TideKV, Fig. 3 and Fig. 5; HillInfer, CEC; HeteroCache, Phase 2).
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from oracle.brute import brute_head


def _rand_head(rng, G, W, S, D, scale=1.0):
    return rng.standard_normal((G * W, D)) * scale, rng.standard_normal((S, D))


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed,G,W,S,D,p,K_l,sink,recent", [
    (0, 1, 1, 9, 3, 1, 4, 1, 1),
    (1, 2, 3, 20, 4, 3, 10, 2, 3),
    (2, 3, 4, 33, 5, 7, 15, 4, 4),
    (3, 2, 5, 17, 8, 5, 9, 0, 5),
    (4, 1, 6, 12, 2, 7, 12, 2, 6),     # K_l = S: keep everything
    (5, 4, 2, 25, 6, 1, 7, 4, 2),
])
def test_oracle_matches_brute_force(seed, G, W, S, D, p, K_l, sink, recent):
    rng = np.random.default_rng(seed)
    q, k = _rand_head(rng, G, W, S, D, scale=1.5)
    a = O.score_head(q, k, W, p)
    idx = O.select_topk(a["s"], K_l, sink, recent)
    b = brute_head(q.tolist(), k.tolist(), W, p, K_l, sink, recent)
    for key in ("m", "Z", "r", "s"):
        np.testing.assert_allclose(a[key], np.array(b[key]), rtol=1e-12, atol=1e-15)
    assert idx.tolist() == b["idx"]


def test_hand_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "hand_example.json")))
    ln2 = math.log(2.0)
    q = np.array(g["q"], dtype=np.float64)
    k = (np.array(g["k_over_ln2"], dtype=np.float64) * ln2)[:, None]
    frac = lambda xs: np.array([float(Fraction(x)) for x in xs])  # noqa: E731
    L = O.dense_logits(q, k, g["W"])
    m, Z = O.lse_normalisers(L)
    np.testing.assert_allclose(m, np.array(g["m_over_ln2"]) * ln2, rtol=1e-14)
    np.testing.assert_allclose(Z, frac(g["Z"]), rtol=1e-14)
    P = O.attention_weights(L, m, Z)
    np.testing.assert_allclose(P, np.array([frac(row) for row in g["P"]]), rtol=1e-14, atol=1e-16)
    r = O.window_group_sum(P)
    np.testing.assert_allclose(r, frac(g["r"]), rtol=1e-14)
    s = O.avg_pool(r, 3)
    np.testing.assert_allclose(s, frac(g["pool_3"]), rtol=1e-14)
    for key in ("select", "select_all"):
        c = g[key]
        sc = O.avg_pool(r, c["pool_k"])
        assert O.select_topk(sc, c["K_l"], c["sink"], c["recent"]).tolist() == c["idx"]


# ------------------------------------------------------------- invariants
@pytest.mark.parametrize("seed,G,W,S,D", [(0, 4, 16, 300, 16), (1, 5, 8, 97, 32), (2, 1, 1, 50, 8)])
def test_weights_sum_to_one_and_mass_is_GW(seed, G, W, S, D):
    rng = np.random.default_rng(seed)
    q, k = _rand_head(rng, G, W, S, D, scale=2.0)
    L = O.dense_logits(q, k, W)
    m, Z = O.lse_normalisers(L)
    P = O.attention_weights(L, m, Z)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-13)
    r = O.window_group_sum(P)
    assert abs(r.sum() - G * W) < 1e-10
    # causal mask: query i puts no weight after its own position t_i
    t = O.window_positions(S, W)
    for a in range(G * W):
        assert np.all(P[a, t[a % W] + 1:] == 0.0)
        assert P[a, t[a % W]] > 0.0


@pytest.mark.parametrize("S,b_s", [(257, 64), (512, 128), (300, 1000), (129, 1)])
def test_two_pass_blockwise_equals_dense(S, b_s):
    rng = np.random.default_rng(S)
    G, W, D, p = 2, 8, 16, 7
    q, k = _rand_head(rng, G, W, S, D, scale=2.0)
    dense = O.score_head(q, k, W, p)
    K_l = 40
    tp = O.two_pass_blockwise(q, k, W, b_s, p, K_l, 4, W)
    np.testing.assert_allclose(tp["m"], dense["m"], rtol=1e-13)
    np.testing.assert_allclose(tp["Z"], dense["Z"], rtol=1e-12)
    assert tp["idx"].tolist() == O.select_topk(dense["s"], K_l, 4, W).tolist()


def test_two_pass_temp_independent_of_S():
    rng = np.random.default_rng(7)
    G, W, D, p, b_s, K_l = 2, 4, 8, 7, 64, 40
    peaks = []
    for S in (1024, 2048, 4096):
        q, k = _rand_head(rng, G, W, S, D)
        peaks.append(O.two_pass_blockwise(q, k, W, b_s, p, K_l, 4, W)["peak_temp"])
    assert peaks[0] == peaks[1] == peaks[2]
    assert peaks[0] < 1024


def test_softmax_special_case_and_raw_dot_ranking():
    """G = W = 1, p = 1: the weights are torch.softmax of the logits, and the
    selection equals top-k of the raw inner products (HillInfer, CEC: the
    softmax is monotone, so ranking by q.k is the same)."""
    rng = np.random.default_rng(11)
    S, D = 200, 32
    q, k = _rand_head(rng, 1, 1, S, D, scale=1.3)
    sc = O.score_head(q, k, 1, 1)
    qt, kt = torch.from_numpy(q), torch.from_numpy(k)
    ref = torch.softmax(torch.matmul(qt, kt.T) / math.sqrt(D), dim=-1)[0].numpy()
    np.testing.assert_allclose(sc["r"], ref, rtol=1e-12)
    sink, recent, K_l = 3, 2, 30
    idx = O.select_topk(sc["s"], K_l, sink, recent)
    raw = (qt @ kt.T)[0]
    raw[:sink] = -float("inf")
    raw[S - recent:] = -float("inf")
    top = torch.topk(raw, K_l - sink - recent).indices.numpy()
    expect = sorted(set(range(sink)) | set(range(S - recent, S)) | set(top.tolist()))
    assert idx.tolist() == expect


@pytest.mark.parametrize("G,W,S,p", [(2, 4, 40, 1), (3, 8, 64, 7)])
def test_all_equal_keys_closed_form(G, W, S, p):
    """Identical keys: P_ij = 1/(t_i + 1) for j <= t_i, and every tie goes to
    the lower index."""
    D = 8
    rng = np.random.default_rng(5)
    q = rng.standard_normal((G * W, D))
    k = np.tile(rng.standard_normal((1, D)), (S, 1))
    L = O.dense_logits(q, k, W)
    m, Z = O.lse_normalisers(L)
    P = O.attention_weights(L, m, Z)
    t = O.window_positions(S, W)
    for a in range(G * W):
        ti = t[a % W]
        np.testing.assert_allclose(P[a, : ti + 1], 1.0 / (ti + 1), rtol=1e-14)
        np.testing.assert_allclose(Z[a], ti + 1, rtol=1e-14)
    r = O.window_group_sum(P)
    expect_r = np.array([G * sum(1.0 / (ti + 1) for ti in t if ti >= j) for j in range(S)])
    np.testing.assert_allclose(r, expect_r, rtol=1e-13)
    sink, recent = 4, W
    n_sel = 10
    idx = O.select_topk(O.avg_pool(r, p), n_sel + sink + recent, sink, recent)
    lo = max(sink, (p - 1) // 2)
    chosen = [j for j in idx.tolist() if sink <= j < S - recent]
    assert chosen == list(range(lo, lo + n_sel))


@pytest.mark.parametrize("p", [1, 3, 5, 7, 9])
def test_avg_pool_against_convolution(p):
    r = np.random.default_rng(p).random(57)
    s = O.avg_pool(r, p)
    np.testing.assert_allclose(s, np.convolve(r, np.ones(p), mode="same") / p, rtol=1e-14)
    if p == 1:
        assert np.array_equal(s, r)


def test_avg_pool_rejects_even_width():
    with pytest.raises(ValueError):
        O.avg_pool(np.ones(5), 4)


# ------------------------------------------------------------- selection
def test_select_invariants_random():
    rng = np.random.default_rng(3)
    for trial in range(50):
        S = int(rng.integers(1, 200))
        sink = int(rng.integers(0, 6))
        recent = int(rng.integers(0, 20))
        R = O.mandatory_set(S, sink, recent)
        K_l = int(rng.integers(len(R), S + 5)) if len(R) <= S + 4 else len(R)
        s = np.round(rng.random(S), 2)             # plenty of exact ties
        idx = O.select_topk(s, K_l, sink, recent)
        assert len(idx) == min(K_l, S)
        assert np.all(np.diff(idx) > 0)
        assert set(R.tolist()) <= set(idx.tolist())
        # every dropped non-mandatory key ranks below every kept one
        kept = [j for j in idx if j not in set(R.tolist())]
        dropped = sorted(set(range(S)) - set(idx.tolist()))
        for d in dropped:
            for c in kept:
                assert (s[c], -c) > (s[d], -d)


def test_select_mandatory_union_and_errors():
    assert O.mandatory_set(10, 4, 8).tolist() == list(range(10))
    assert O.mandatory_set(10, 2, 3).tolist() == [0, 1, 7, 8, 9]
    assert O.mandatory_set(10, 0, 0).tolist() == []
    with pytest.raises(ValueError):
        O.select_topk(np.ones(10), 4, 2, 3)
    assert O.select_topk(np.ones(10), 12, 2, 3).tolist() == list(range(10))


def test_gather_golden_position_rows(golden_dir):
    """K/V rows that encode their own position come back in selection order."""
    import torch
    g = json.load(open(os.path.join(golden_dir, "gather_positions.json")))
    S, D = g["S"], g["D"]
    j = torch.arange(S, dtype=torch.float32)
    k = torch.stack([j, -j], dim=1).to(torch.bfloat16)
    v = torch.stack([100 + j, -100 - j], dim=1).to(torch.bfloat16)
    assert k.shape == (S, D)
    kh, vh, pos = O.gather(k, v, np.array(g["idx"]))
    assert kh.dtype == torch.bfloat16 and vh.dtype == torch.bfloat16
    assert kh.float().tolist() == g["k_hat"]
    assert vh.float().tolist() == g["v_hat"]
    assert pos.dtype == np.int32 and pos.tolist() == g["pos"]


def test_compress_layer_rows_are_the_selected_positions():
    """The retained rows of a whole compress are the rows at its own (ascending) positions."""
    import torch
    rng = np.random.default_rng(3)
    B, Hq, Hkv, S, D, W = 1, 4, 2, 48, 4, 4
    q = torch.from_numpy(rng.standard_normal((B, Hq, W, D))).to(torch.bfloat16)
    j = torch.arange(S, dtype=torch.float32)[:, None]
    noise = torch.from_numpy(rng.standard_normal((B, Hkv, S, D - 1))).float()
    k = torch.cat([j.expand(B, Hkv, S, 1), noise], dim=3).to(torch.bfloat16)   # column 0 = position
    v = (-1 - j).expand(B, Hkv, S, D).to(torch.bfloat16)                      # exact: |v| <= 256
    out = O.compress_layer(q, k, v, [10, 17], 2, 4, 3)
    for (b, h), r in out.items():
        pos = r["pos"].tolist()
        assert pos == sorted(set(pos)) and len(pos) == [10, 17][h]
        assert r["k_hat"][:, 0].float().tolist() == pos
        assert r["v_hat"][:, 0].float().tolist() == [-1 - p for p in pos]


def test_gqa_head_map_hand_case():
    """Hand-built GQA case: the scores follow from the head map g -> g // G.

    H_q=4, H_kv=2 (G=2), W=1, D=2, S=8.  KV head 0 has one non-zero key, at
    position 3, equal to (c, 0); KV head 1 has one, at position 5, equal to
    (0, c); c = 4*sqrt(2), so q.k/sqrt(D) = 4 for an aligned query.  Query
    heads 0 and 1 are (1, 0), heads 2 and 3 are (0, 1).  With contiguous
    groups each KV head sees two aligned queries, so for the single window
    query (t = 7, all keys visible) the heavy key gets 2 e^4 / (e^4 + 7) and
    every other key 2 / (e^4 + 7).  Any other map puts an orthogonal query
    (uniform weights 1/8) in the group.
    """
    S, D, W = 8, 2, 1
    c = 4 * math.sqrt(2)
    k = np.zeros((1, 2, S, D))
    k[0, 0, 3] = (c, 0.0)
    k[0, 1, 5] = (0.0, c)
    q = np.zeros((1, 4, W, D))
    q[0, 0:2, 0] = (1.0, 0.0)
    q[0, 2:4, 0] = (0.0, 1.0)
    out = O.compress_layer(q, k, np.zeros_like(k), [3, 3], 1, 1, 1)
    den = math.exp(4) + 7
    for h, heavy in ((0, 3), (1, 5)):
        want = np.full(S, 2 / den)
        want[heavy] = 2 * math.exp(4) / den
        np.testing.assert_allclose(out[(0, h)]["r"], want, rtol=1e-13)
        assert out[(0, h)]["idx"].tolist() == sorted({0, heavy, 7})


# --------------------------------------------------- closed forms from pages
def test_retained_cache_is_512_mib(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "retained_cache_512mib.json")))
    got = O.retained_cache_bytes(g["N"], g["H_kv"], g["K_l"], g["D"], g["B"], g["elem_bytes"])
    assert got == g["bytes"] == g["mib"] * 2**20


def test_inverse_stability_budgets():
    s = np.array([0.8307, 0.2256, 0.3952, 0.9737, 0.7709, 0.4175, 0.3023, 0.9045])
    total = round(0.3 * 32768 * 8)
    assert total == 78643
    K = O.budgets_inverse_stability(s, total, 68, 32768)
    assert int(K.sum()) == total
    exact = total * (1 / s) / (1 / s).sum()
    assert np.all(np.abs(K - exact) < 1.0)
    # unstable heads (small s) get larger budgets
    assert np.all(np.diff(K[np.argsort(s)]) <= 0)
    # clamps
    K2 = O.budgets_inverse_stability(np.array([1.0, 1.0, 0.01]), 300, 50, 200)
    assert K2.tolist() == [50, 50, 200]
    # largest remainder, ties to the lower head index
    assert O.budgets_inverse_stability(np.ones(3), 10, 0, 100).tolist() == [4, 3, 3]
    # worked by hand: s = (1, 2, 4) -> w = (1, 1/2, 1/4), shares 10 w / (7/4) =
    # (40/7, 20/7, 10/7); floors (5, 2, 1) leave 2; remainders (5/7, 6/7, 3/7)
    # give them to heads 1 and 0
    assert O.budgets_inverse_stability(np.array([1.0, 2.0, 4.0]), 10, 0, 100).tolist() == [6, 3, 1]


def test_retained_layout():
    off = O.retained_layout(100, [10, 200, 5])
    assert off.tolist() == [0, 10, 110, 115]


def test_compress_layer_gqa_head_map():
    """Query head g belongs to KV head g // G (contiguous groups)."""
    rng = np.random.default_rng(9)
    B, Hq, Hkv, S, D, W = 2, 6, 2, 40, 8, 3
    q = rng.standard_normal((B, Hq, W, D))
    k = rng.standard_normal((B, Hkv, S, D))
    v = rng.standard_normal((B, Hkv, S, D))
    out = O.compress_layer(q, k, v, [12, 20], 2, 3, 3)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            ref = O.score_head(q[b, h * G:(h + 1) * G].reshape(G * W, D), k[b, h], W, 3)
            np.testing.assert_allclose(out[(b, h)]["s"], ref["s"], rtol=1e-14)
            assert len(out[(b, h)]["idx"]) == [12, 20][h]
            assert np.array_equal(out[(b, h)]["k_hat"], k[b, h][out[(b, h)]["idx"]])
