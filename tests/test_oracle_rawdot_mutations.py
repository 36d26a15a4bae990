"""Planted mistakes in the INT8 raw-product oracle must be caught by its pins
(CPU only).

Each mutant replaces one function of oracle/rawdot_int8.py with a plausible
wrong variant (another rounding rule, a wrong scale, a dropped factor, a
mean instead of a sum) and checks that at least one pin of
tests/test_oracle_rawdot.py fails on it.
"""

import os

import numpy as np
import pytest

from oracle import rawdot_int8 as R
import tests.test_oracle_rawdot as pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(pins.__file__)), "golden")


def _suite():
    """Run the pins; return the number that failed."""
    checks = [
        lambda: pins.test_hand_example(GOLDEN),
        lambda: pins.test_round_half_to_even_hand_case(GOLDEN),
        lambda: pins.test_codes_span_and_zero_rows(),
        lambda: pins.test_summed_query_is_the_softmax_free_window_group_sum(1, 2, 4, 64, 16),
        lambda: pins.test_int8_scores_within_the_rounding_bound(0, 1.0),
        lambda: pins.test_int8_scores_within_the_rounding_bound(2, 30.0),
        lambda: pins.test_row_batched_scores_equal_the_per_key_ones(),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, ValueError, IndexError, ZeroDivisionError, FloatingPointError):
            failed += 1
    return failed


def test_unmutated_rawdot_oracle_passes_suite():
    assert _suite() == 0


def _quantize_with(round_fn, num=127.0, amax_fn=None, invert_scale=False):
    def q(x):
        x = R._f32(x)
        amax = np.float32(amax_fn(x) if amax_fn else np.max(np.abs(x))) if x.size else np.float32(0.0)
        if amax == 0:
            return np.zeros(x.shape, dtype=np.int32), np.float32(0.0)
        inv = np.float32(np.float32(num) / amax)
        codes = np.clip(round_fn((x * inv).astype(np.float32)).astype(np.int32), -127, 127)
        scale = np.float32(np.float32(127.0) / amax) if invert_scale else np.float32(amax / np.float32(127.0))
        return codes, scale
    return q


def _round_half_away(y):
    return np.sign(y) * np.floor(np.abs(y) + 0.5)


def _round_half_up(y):
    return np.floor(y + 0.5)


def _summed_query_mean(q_grp):
    q = R._f32(q_grp)
    return (q.sum(axis=0, dtype=np.float32) / np.float32(q.shape[0])).astype(np.float32)


def _summed_query_drops_last_row(q_grp):
    q = R._f32(q_grp)
    acc = np.zeros(q.shape[1], dtype=np.float32)
    for r in range(q.shape[0] - 1):
        acc = (acc + q[r]).astype(np.float32)
    return acc


def _scores_query_scale_twice(q_grp, k):
    qc, sq = R.quantize_int8(R.summed_query(q_grp))
    kk = R._f32(k)
    out = np.empty(kk.shape[0], dtype=np.float32)
    for j in range(kk.shape[0]):
        kc, _ = R.quantize_int8(kk[j])
        dot = int(np.dot(qc.astype(np.int64), kc.astype(np.int64)))
        out[j] = np.float32(np.float32(np.float32(dot) * sq) * sq)
    return out


def _scores_without_query_scale(q_grp, k):
    qc, _ = R.quantize_int8(R.summed_query(q_grp))
    kk = R._f32(k)
    out = np.empty(kk.shape[0], dtype=np.float32)
    for j in range(kk.shape[0]):
        kc, sk = R.quantize_int8(kk[j])
        dot = int(np.dot(qc.astype(np.int64), kc.astype(np.int64)))
        out[j] = np.float32(np.float32(dot) * sk)
    return out


MUTANTS = {
    "round half away from zero": ("quantize_int8", _quantize_with(_round_half_away)),
    "round half up": ("quantize_int8", _quantize_with(_round_half_up)),
    "truncate": ("quantize_int8", _quantize_with(np.trunc)),
    "255 levels": ("quantize_int8", _quantize_with(np.rint, num=255.0)),
    "inverted scale": ("quantize_int8", _quantize_with(np.rint, invert_scale=True)),
    "mean |x| as the range": ("quantize_int8", _quantize_with(np.rint, amax_fn=lambda x: np.mean(np.abs(x)))),
    "query mean instead of sum": ("summed_query", _summed_query_mean),
    "query sum drops the last row": ("summed_query", _summed_query_drops_last_row),
    "query scale used for the key": ("raw_scores_int8", _scores_query_scale_twice),
    "no query scale": ("raw_scores_int8", _scores_without_query_scale),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_rawdot_mutant_is_caught(name, monkeypatch):
    fn_name, mutant = MUTANTS[name]
    monkeypatch.setattr(R, fn_name, mutant)
    with np.errstate(all="ignore"):
        assert _suite() > 0, f"mutant '{name}' passes every pin"
