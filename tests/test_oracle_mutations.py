"""Planted mistakes in the oracle must be caught by the pins (CPU only).

Each mutant replaces one oracle function with a plausible wrong variant (a
dropped term, a wrong sign or index, a wrong divisor, the wrong tie-break) and
checks that at least one pin of tests/test_oracle_pins.py fails on it.
"""

import math

import numpy as np
import pytest

from oracle import kvc_oracle as O
import tests.test_oracle_pins as pins

GOLDEN = pins.os.path.join(pins.os.path.dirname(pins.os.path.abspath(pins.__file__)), "golden")


def _suite():
    """Run the pins; return the number that failed."""
    checks = [
        lambda: pins.test_oracle_matches_brute_force(1, 2, 3, 20, 4, 3, 10, 2, 3),
        lambda: pins.test_oracle_matches_brute_force(2, 3, 4, 33, 5, 7, 15, 4, 4),
        lambda: pins.test_hand_worked_example(GOLDEN),
        lambda: pins.test_weights_sum_to_one_and_mass_is_GW(0, 4, 16, 300, 16),
        lambda: pins.test_all_equal_keys_closed_form(3, 8, 64, 7),
        lambda: pins.test_avg_pool_against_convolution(7),
        lambda: pins.test_select_invariants_random(),
        lambda: pins.test_softmax_special_case_and_raw_dot_ranking(),
        lambda: pins.test_inverse_stability_budgets(),
        lambda: pins.test_gather_golden_position_rows(GOLDEN),
        lambda: pins.test_compress_layer_rows_are_the_selected_positions(),
        lambda: pins.test_gqa_head_map_hand_case(),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    return failed


def test_unmutated_oracle_passes_suite():
    assert _suite() == 0


def _logits_scale_1_over_D(q_grp, k, W):
    q_grp, k = O.as_f64(q_grp), O.as_f64(k)
    S, D = k.shape
    L = (q_grp @ k.T) / D
    t = O.window_positions(S, W)[np.arange(q_grp.shape[0]) % W]
    L[np.arange(S)[None, :] > t[:, None]] = -np.inf
    return L


def _logits_mask_off_by_one(q_grp, k, W):
    q_grp, k = O.as_f64(q_grp), O.as_f64(k)
    S, D = k.shape
    L = (q_grp @ k.T) / math.sqrt(D)
    t = O.window_positions(S, W)[np.arange(q_grp.shape[0]) % W]
    L[np.arange(S)[None, :] >= t[:, None]] = -np.inf
    return L


def _logits_rows_grouped_wrong(q_grp, k, W):
    q_grp, k = O.as_f64(q_grp), O.as_f64(k)
    S, D = k.shape
    rows = q_grp.shape[0]
    G = rows // W
    L = (q_grp @ k.T) / math.sqrt(D)
    t = O.window_positions(S, W)[np.arange(rows) // G]      # (i, g) order instead of (g, i)
    L[np.arange(S)[None, :] > t[:, None]] = -np.inf
    return L


def _logits_no_causal_mask(q_grp, k, W):
    q_grp, k = O.as_f64(q_grp), O.as_f64(k)
    return (q_grp @ k.T) / math.sqrt(k.shape[1])


def _lse_without_max(L):
    m = L.max(axis=1)
    return m, np.exp(L).sum(axis=1)


def _weights_sign_flip(L, m, Z):
    return np.exp(m[:, None] - L) / Z[:, None]


def _group_mean(P):
    return P.mean(axis=0)


def _pool_divisor_in_range(r, p):
    S = len(r)
    h = (p - 1) // 2
    return np.array([np.mean(r[max(0, j - h):min(S, j + h + 1)]) for j in range(S)])


def _pool_off_centre(r, p):
    s = np.convolve(r, np.ones(p), mode="full")[: len(r)] / p
    return s


def _select_tie_to_higher_index(s, K_l, sink, recent):
    s = np.asarray(s)
    S = len(s)
    R = O.mandatory_set(S, sink, recent)
    if K_l < len(R):
        raise ValueError
    if K_l >= S:
        return np.arange(S)
    cand = np.setdiff1d(np.arange(S), R)
    order = np.lexsort((-cand, -s[cand]))
    return np.sort(np.concatenate([R, cand[order[: K_l - len(R)]]]))


def _select_drops_sink(s, K_l, sink, recent):
    return O.__dict__["_orig_select"](s, K_l, 0, recent)


def _window_shifted(S, W):
    return np.arange(S - W - 1, S - 1)


def _budget_proportional_to_s(s_stable, total, lo, hi):
    s = np.asarray(s_stable, dtype=np.float64)
    exact = total * s / s.sum()
    base = np.floor(exact).astype(np.int64)
    base[: int(total - base.sum())] += 1
    return np.clip(base, lo, hi).astype(np.int32)


def _gather_off_by_one(k, v, idx):
    idx = np.minimum(np.asarray(idx, dtype=np.int64) + 1, len(k) - 1)
    return k[idx], v[idx], idx.astype(np.int32)


def _gather_reversed(k, v, idx):
    idx = np.asarray(idx, dtype=np.int64)[::-1].copy()
    return k[idx], v[idx], idx.astype(np.int32)


def _gather_swaps_kv(k, v, idx):
    idx = np.asarray(idx, dtype=np.int64)
    return v[idx], k[idx], idx.astype(np.int32)


def _head_map_modulo(q_b, h, G):
    Hq, W, D = q_b.shape
    Hkv = Hq // G
    return q_b[[g for g in range(Hq) if g % Hkv == h]].reshape(G * W, D)


MUTANTS = {
    "gather_off_by_one": ("gather", _gather_off_by_one),
    "gather_reversed": ("gather", _gather_reversed),
    "gather_swaps_kv": ("gather", _gather_swaps_kv),
    "head_map_modulo": ("group_queries", _head_map_modulo),
    "scale_1_over_D": ("dense_logits", _logits_scale_1_over_D),
    "mask_off_by_one": ("dense_logits", _logits_mask_off_by_one),
    "rows_grouped_wrong": ("dense_logits", _logits_rows_grouped_wrong),
    "no_causal_mask": ("dense_logits", _logits_no_causal_mask),
    "lse_without_max": ("lse_normalisers", _lse_without_max),
    "weights_sign_flip": ("attention_weights", _weights_sign_flip),
    "group_mean": ("window_group_sum", _group_mean),
    "pool_divisor_in_range": ("avg_pool", _pool_divisor_in_range),
    "pool_off_centre": ("avg_pool", _pool_off_centre),
    "tie_to_higher_index": ("select_topk", _select_tie_to_higher_index),
    "drops_sink": ("select_topk", _select_drops_sink),
    "window_shifted": ("window_positions", _window_shifted),
    "budget_prop_to_s": ("budgets_inverse_stability", _budget_proportional_to_s),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    fn_name, mutant = MUTANTS[name]
    monkeypatch.setitem(O.__dict__, "_orig_select", O.select_topk)
    monkeypatch.setattr(O, fn_name, mutant)
    assert _suite() > 0, f"mutant {name} passed every pin"
