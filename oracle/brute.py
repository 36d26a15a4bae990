"""Pure-Python brute force of the layer-end scorer for tiny shapes.

TEST INFRASTRUCTURE: a second, loop-by-loop statement of the same definition
as ``kvc_oracle`` (TideKV, Fig. 3), with ``math.exp`` and Python floats and no
NumPy, used to pin the fp64 oracle on tiny inputs.  Keep S*G*W*D small.
"""

from __future__ import annotations

import math


def brute_head(q_grp, k, W, pool_k, K_l, sink, recent):
    """q_grp: list of G*W rows (lists of D floats), row g*W+i; k: list of S rows."""
    S = len(k)
    D = len(k[0])
    rows = len(q_grp)
    m, Z = [], []
    P = [[0.0] * S for _ in range(rows)]
    for a in range(rows):
        t = S - W + (a % W)
        logit = []
        for j in range(S):
            if j > t:
                logit.append(None)
                continue
            dot = 0.0
            for d in range(D):
                dot += q_grp[a][d] * k[j][d]
            logit.append(dot / math.sqrt(D))
        mx = max(x for x in logit if x is not None)
        z = 0.0
        for x in logit:
            if x is not None:
                z += math.exp(x - mx)
        m.append(mx)
        Z.append(z)
        for j, x in enumerate(logit):
            P[a][j] = 0.0 if x is None else math.exp(x - mx) / z
    r = [sum(P[a][j] for a in range(rows)) for j in range(S)]
    h = (pool_k - 1) // 2
    s = []
    for j in range(S):
        acc = 0.0
        for d in range(-h, h + 1):
            if 0 <= j + d < S:
                acc += r[j + d]
        s.append(acc / pool_k)
    mand = [j for j in range(S) if j < sink or j >= S - recent]
    if K_l >= S:
        idx = list(range(S))
    else:
        n_sel = K_l - len(mand)
        others = [j for j in range(S) if not (j < sink or j >= S - recent)]
        # selection by repeated arg-max: highest score, lowest index on ties
        chosen = []
        pool = list(others)
        for _ in range(n_sel):
            best = None
            for j in pool:
                if best is None or s[j] > s[best]:
                    best = j
            chosen.append(best)
            pool.remove(best)
        idx = sorted(mand + chosen)
    return {"m": m, "Z": Z, "r": r, "s": s, "idx": idx}
