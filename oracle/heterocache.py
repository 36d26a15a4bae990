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

Pins (tests/test_oracle_heterocache.py): closed forms (identical, disjoint,
nested sets), symmetry, the range [0, 1], a hand-worked example, and the
similarity as the row maximum of the pairwise matrix.
"""

from __future__ import annotations

import numpy as np

__all__ = ["overlap_coefficient", "head_similarity"]


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
