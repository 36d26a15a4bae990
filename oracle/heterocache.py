"""CPU oracle for HeteroCache's overlap measurements (test infrastructure).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import this module.  It shares no code with the CUDA
library and imports nothing from it.

HeteroCache ("Key Contributions" 1; "Methodology", Phase 1) measures how
much two top-k attention sets agree by the overlap coefficient
|A n B| / min(|A|, |B|): the stability score compares a head's decoding
top-k with its prefill set, the similarity score takes, per head, the
largest overlap with any other head of the same layer.

Readings: sets are sets of positions (duplicates collapse); the ratio is one
float32 division of the two exact integers; an empty set gives 0; with a
single head the similarity is 0.  The budgets of Phase 2 are
``kvc_oracle.budgets_inverse_stability``.

Phase 1 scores over decoding steps: the stability score of a head is the
median, over T steps, of the overlap between its top-k at step t and its
prefill set; the similarity score is the median, over the same steps, of the
per-step maximum overlap with another head of the layer.  Reading of
"median": the middle value of the T fp32 per-step overlaps for odd T; for
even T the mean of the two middle values, (a + b) / 2 formed exactly (in
fp64) and rounded once to fp32 (-0 counts as +0).

Pins (tests/test_oracle_heterocache.py): closed forms (identical, disjoint,
nested sets), symmetry, the range [0, 1], a hand-worked example, the
similarity as the row maximum of the pairwise matrix, hand-worked medians of
odd and even T, and the medians against an exact rational brute force.
"""

from __future__ import annotations

import numpy as np

__all__ = ["overlap_coefficient", "head_similarity", "median_over_steps", "stability_over_steps",
           "similarity_over_steps"]


def overlap_coefficient(a, b) -> np.float32:
    sa, sb = set(int(x) for x in a), set(int(x) for x in b)
    mn = min(len(sa), len(sb))
    if mn == 0:
        return np.float32(0.0)
    return np.float32(np.float32(len(sa & sb)) / np.float32(mn))


def head_similarity(sets) -> np.ndarray:
    """sets: list of H index collections -> fp32 [H], max over j != i."""
    H = len(sets)
    out = np.zeros(H, dtype=np.float32)
    for i in range(H):
        best = np.float32(0.0)
        for j in range(H):
            if j != i:
                best = max(best, overlap_coefficient(sets[i], sets[j]))
        out[i] = best
    return out


def median_over_steps(x) -> np.ndarray:
    """x: fp32 [T, H] per-step values -> fp32 [H], the median over the steps."""
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    out = np.zeros(H, dtype=np.float32)
    for h in range(H):
        v = np.sort(x[:, h].astype(np.float64) + 0.0)      # -0 counts as +0
        if T % 2:
            out[h] = np.float32(v[T // 2])
        else:
            out[h] = np.float32((v[T // 2 - 1] + v[T // 2]) / 2.0)
    return out


def stability_over_steps(dec_sets, pre_sets):
    """dec_sets[t][h]: head h's top-k at decoding step t; pre_sets[h]: its
    prefill set.  Returns (per-step overlaps fp32 [T, H], stability [H])."""
    T, H = len(dec_sets), len(pre_sets)
    per = np.zeros((T, H), dtype=np.float32)
    for t in range(T):
        for h in range(H):
            per[t, h] = overlap_coefficient(dec_sets[t][h], pre_sets[h])
    return per, median_over_steps(per)


def similarity_over_steps(step_sets):
    """step_sets[t][h]: head h's top-k at step t (one layer).  Returns
    (per-step maximum overlaps fp32 [T, H], similarity [H])."""
    per = np.stack([head_similarity(sets) for sets in step_sets]).astype(np.float32)
    return per, median_over_steps(per)
