"""CPU oracle (fp64 NumPy) for layer-end KV-cache compression by attention scoring.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library and imports nothing from it.

What it computes is the plain definition that TideKV's memory-controlled
two-pass blockwise scorer reaches exactly, up to rounding (TideKV,
"Memory-controlled two-pass blockwise scoring", Fig. 3): the scorer avoids
materialising the dense W x S observation-by-prefix score tensor, so the
oracle materialises it.  Per batch element b and KV head h, with G = H_q/H_kv
query heads sharing h (query head g belongs to KV head g // G):

1. logits   L[(g,i), j] = q_{g,i} . k_j / sqrt(D) for j <= t_i, else -inf,
            where t_i = S - W + i is the absolute position of window query i;
2. normalisers m = max_j L, Z = sum_j exp(L - m) per query row (Fig. 3: the
            numerically stable log-sum-exp normalisers (m_q, Z_q));
3. weights  P = exp(L - m) / Z;
4. r_j      = sum over the window queries and the GQA group of P[:, j];
5. s_j      = centred, zero-padded average pool of r with width p;
6. R_mand   = sink keys [0, sink) and recent keys [S - recent, S);
            keep the top (K_l - |R_mand|) non-mandatory keys by
            (s descending, index ascending), together with R_mand (Fig. 3);
7. gather   retained K, V rows and their absolute positions (Fig. 2).

Readings where the pages are silent: the window is the last W prompt
positions; each window query attends causally (j <= t_i); scores are summed,
not averaged, over the group; pooling is a centred average with zero padding
and divisor p; ties go to the lower index; retained entries are listed in
ascending position order.

Functions and their pins (tests/test_oracle_pins.py):
  dense_logits, lse_normalisers, attention_weights, window_group_sum:
      brute force, hand-worked example, G=W=1 softmax, all-equal keys,
      row sums = 1, sum r = G*W.
  avg_pool: brute force, hand example, k=1 identity, np.convolve.
  mandatory_set, select_topk: brute force, raw-dot-product special case,
      all-equal ties, |kept| = min(K_l, S), R_mand kept.
  gather: position-encoding rows (golden), order and off-by-one.
  group_queries: hand-built GQA case whose scores follow from the head map.
  two_pass_blockwise: equals the dense path; temp independent of S.
  budgets_inverse_stability: exact-rational shares; sums, proportionality,
      clamps, a hand-worked largest-remainder case.
  retained_cache_bytes: 512 MiB at TideKV's main setting.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

__all__ = [
    "as_f64", "window_positions", "dense_logits", "lse_normalisers",
    "attention_weights", "window_group_sum", "avg_pool", "score_head", "group_queries",
    "mandatory_set", "select_topk", "gather", "compress_layer",
    "two_pass_blockwise", "budgets_inverse_stability", "retained_layout",
    "retained_cache_bytes",
]


def as_f64(x) -> np.ndarray:
    """Exact conversion of a bf16/fp32 tensor or array to fp64."""
    try:
        import torch  # only for the conversion of torch inputs
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def window_positions(S: int, W: int) -> np.ndarray:
    """t_i = S - W + i: the observation window is the last W prompt positions."""
    if not 1 <= W <= S:
        raise ValueError("need 1 <= W <= S")
    return np.arange(S - W, S, dtype=np.int64)


def dense_logits(q_grp: np.ndarray, k: np.ndarray, W: int) -> np.ndarray:
    """Dense observation-by-prefix logits for one KV head (TideKV, Fig. 3).

    q_grp: [G*W, D] window queries of the group, row index g*W + i.
    k:     [S, D] prefix keys of the KV head.
    Returns L [G*W, S] fp64 with -inf where key j lies after query i (j > t_i).
    The 1/sqrt(D) scale is the one of rho(Q K^T / sqrt(d)) (HillInfer, CEC).
    """
    q_grp = as_f64(q_grp)
    k = as_f64(k)
    S, D = k.shape
    rows = q_grp.shape[0]
    L = (q_grp @ k.T) / math.sqrt(D)
    t = window_positions(S, W)[np.arange(rows) % W]
    L[np.arange(S)[None, :] > t[:, None]] = -np.inf
    return L


def lse_normalisers(L: np.ndarray):
    """Per-row log-sum-exp normalisers (m_q, Z_q) of TideKV Fig. 3."""
    m = L.max(axis=1)
    Z = np.exp(L - m[:, None]).sum(axis=1)
    return m, Z


def attention_weights(L: np.ndarray, m: np.ndarray, Z: np.ndarray) -> np.ndarray:
    """Normalised weights P = exp(L - m) / Z (pass 2 of TideKV Fig. 3)."""
    return np.exp(L - m[:, None]) / Z[:, None]


def window_group_sum(P: np.ndarray) -> np.ndarray:
    """r_j: the weights summed over the window queries and the GQA group."""
    return P.sum(axis=0)


def avg_pool(r: np.ndarray, p: int) -> np.ndarray:
    """Centred average pool of width p (odd), zero padding, divisor always p."""
    if p < 1 or p % 2 == 0:
        raise ValueError("pool width must be odd and >= 1")
    r = np.asarray(r, dtype=np.float64)
    S = r.shape[0]
    h = (p - 1) // 2
    padded = np.concatenate([np.zeros(h), r, np.zeros(h)])
    s = np.zeros(S)
    for d in range(p):
        s += padded[d:d + S]
    return s / p


def score_head(q_grp, k, W: int, pool_k: int) -> dict:
    """m, Z (natural-log units), r and pooled s for one (b, KV head)."""
    L = dense_logits(q_grp, k, W)
    m, Z = lse_normalisers(L)
    P = attention_weights(L, m, Z)
    r = window_group_sum(P)
    return {"m": m, "Z": Z, "r": r, "s": avg_pool(r, pool_k)}


def mandatory_set(S: int, sink: int, recent: int) -> np.ndarray:
    """R_mand: the sink keys [0, sink) and the recent keys [S-recent, S), sorted."""
    if sink < 0 or recent < 0:
        raise ValueError("sink/recent must be >= 0")
    mask = np.zeros(S, dtype=bool)
    mask[: min(sink, S)] = True
    mask[max(S - recent, 0):] = True
    return np.nonzero(mask)[0]


def select_topk(s: np.ndarray, K_l: int, sink: int, recent: int) -> np.ndarray:
    """Retained positions for one head, ascending (TideKV Fig. 3).

    Keeps R_mand plus the top (K_l - |R_mand|) non-mandatory keys ordered by
    (score descending, index ascending).  If K_l >= S every key is kept.
    Raises ValueError if K_l < |R_mand|.
    """
    s = np.asarray(s)
    S = s.shape[0]
    R = mandatory_set(S, sink, recent)
    if K_l < len(R):
        raise ValueError("budget smaller than the mandatory set")
    if K_l >= S:
        return np.arange(S, dtype=np.int64)
    n_sel = K_l - len(R)
    cand = np.setdiff1d(np.arange(S), R)
    order = np.lexsort((cand, -s[cand]))      # primary -s, secondary index
    chosen = cand[order[:n_sel]]
    return np.sort(np.concatenate([R, chosen])).astype(np.int64)


def gather(k, v, idx):
    """Retained (K_hat, V_hat) rows and their absolute positions (TideKV Fig. 2)."""
    idx = np.asarray(idx, dtype=np.int64)
    return k[idx], v[idx], idx.astype(np.int32)


def group_queries(q_b: np.ndarray, h: int, G: int) -> np.ndarray:
    """Window queries of KV head h as one [G*W, D] block, row g*W + i.

    GQA with contiguous groups: query heads h*G .. h*G + G - 1 share KV head
    h, i.e. query head g reads KV head g // G.  q_b is [H_q, W, D].
    """
    Hq, W, D = q_b.shape
    return q_b[h * G:(h + 1) * G].reshape(G * W, D)


def compress_layer(q_win, k, v, K_l, sink: int, recent: int, pool_k: int,
                   heads=None) -> dict:
    """The whole layer-end compress for one layer.

    q_win [B, H_q, W, D], k/v [B, H_kv, S, D] (numpy or torch; k/v are gathered
    in their own dtype, so bf16 bytes stay bf16), K_l [H_kv] budgets.
    ``heads``: optional list of (b, h) to compute; default all.
    Returns per-(b, h) dicts with m, Z ([G*W]), r, s ([S]), idx, k_hat, v_hat, pos.
    """
    B, Hq, W, D = q_win.shape
    Hkv, S = k.shape[1], k.shape[2]
    if Hq % Hkv:
        raise ValueError("H_q must be a multiple of H_kv")
    G = Hq // Hkv
    qf = as_f64(q_win)
    out = {}
    for (b, h) in (heads if heads is not None else
                   [(b, h) for b in range(B) for h in range(Hkv)]):
        q_grp = group_queries(qf[b], h, G)
        sc = score_head(q_grp, k[b, h], W, pool_k)
        idx = select_topk(sc["s"], int(K_l[h]), sink, recent)
        kh, vh, pos = gather(k[b, h], v[b, h], idx)
        sc.update(idx=idx, k_hat=kh, v_hat=vh, pos=pos)
        out[(b, h)] = sc
    return out


def two_pass_blockwise(q_grp, k, W: int, b_s: int, pool_k: int, K_l: int,
                       sink: int, recent: int) -> dict:
    """The memory-controlled two-pass scan of TideKV Fig. 3, step by step.

    Pass 1 walks the key blocks of b_s keys and keeps only the running
    (m_q, Z_q) per window query.  Pass 2 walks the blocks again, forms the
    normalised weights, sums them per key, pools them and keeps a running
    candidate list of at most K_l - |R_mand| non-mandatory keys.  Nothing of
    length S is held besides the inputs; ``peak_temp`` counts the largest
    number of temporary values alive at once (a logit tile, the W-length
    state, the pooling carry and the candidate list).
    """
    qf = as_f64(q_grp)
    kf = as_f64(k)
    S, D = kf.shape
    rows = qf.shape[0]
    t = window_positions(S, W)[np.arange(rows) % W]
    scale = 1.0 / math.sqrt(D)
    h = (pool_k - 1) // 2
    R = mandatory_set(S, sink, recent)
    is_mand = lambda j: j < sink or j >= S - recent  # noqa: E731
    if K_l < len(R):
        raise ValueError("budget smaller than the mandatory set")
    n_sel = K_l - len(R)
    peak = 0

    # pass 1: online normalisers
    m = np.full(rows, -np.inf)
    Z = np.zeros(rows)
    for j0 in range(0, S, b_s):
        j1 = min(j0 + b_s, S)
        tile = (qf @ kf[j0:j1].T) * scale
        tile[np.arange(j0, j1)[None, :] > t[:, None]] = -np.inf
        m_new = np.maximum(m, tile.max(axis=1))
        Z = Z * np.exp(m - m_new) + np.exp(tile - m_new[:, None]).sum(axis=1)
        m = m_new
        peak = max(peak, tile.size + 2 * rows)

    # pass 2: weights -> per-key mass -> pooled score -> running top list
    r_hist = {}            # r_j kept only while a pooled score still needs it
    cand_s = np.zeros(0)
    cand_j = np.zeros(0, dtype=np.int64)
    next_out = 0           # next key whose pooled score is due
    for j0 in range(0, S, b_s):
        j1 = min(j0 + b_s, S)
        tile = (qf @ kf[j0:j1].T) * scale
        tile[np.arange(j0, j1)[None, :] > t[:, None]] = -np.inf
        P = np.exp(tile - m[:, None]) / Z[:, None]
        r_blk = P.sum(axis=0)
        for jj in range(j0, j1):
            r_hist[jj] = r_blk[jj - j0]
        # every key whose whole pooling neighbourhood has been seen is due
        last_due = S - 1 if j1 == S else j1 - 1 - h
        new_s, new_j = [], []
        for j in range(next_out, last_due + 1):
            acc = 0.0
            for d in range(-h, h + 1):
                acc += r_hist.get(j + d, 0.0)
            if not is_mand(j):
                new_s.append(acc / pool_k)
                new_j.append(j)
        next_out = last_due + 1
        for jj in [x for x in r_hist if x < next_out - h]:
            del r_hist[jj]
        cand_s = np.concatenate([cand_s, np.asarray(new_s)])
        cand_j = np.concatenate([cand_j, np.asarray(new_j, dtype=np.int64)])
        peak = max(peak, tile.size + 2 * rows + len(r_hist) + 2 * len(cand_s))
        if len(cand_s) > n_sel:
            order = np.lexsort((cand_j, -cand_s))[:n_sel]
            cand_s, cand_j = cand_s[order], cand_j[order]
    if K_l >= S:
        idx = np.arange(S, dtype=np.int64)
    else:
        idx = np.sort(np.concatenate([R, cand_j])).astype(np.int64)
    return {"m": m, "Z": Z, "idx": idx, "peak_temp": peak}


def budgets_inverse_stability(s_stable, total: int, lo: int, hi: int) -> np.ndarray:
    """Per-KV-head budgets l_i proportional to w_i = 1 / s_i (HeteroCache, Phase 2).

    The pages do not print the L_base formula; the reading taken: every head
    is compressed (no full heads), the shares total * w_i / sum(w) are
    rounded by largest remainder (ties to the lower head index) so that they
    sum to ``total``, then clamped to [lo, hi] without redistribution.  The
    shares and their remainders are exact rationals (each fp64 score is
    converted exactly), so the rounding decision involves no floating-point
    error at all.
    """
    s = [Fraction(float(x)) for x in np.asarray(s_stable, dtype=np.float64)]
    if any(x <= 0 for x in s):
        raise ValueError("stability scores must be > 0")
    w = [1 / x for x in s]
    wsum = sum(w, Fraction(0))
    exact = [Fraction(int(total)) * x / wsum for x in w]
    base = [math.floor(x) for x in exact]
    short = int(total - sum(base))
    rem = [x - b for x, b in zip(exact, base)]
    order = sorted(range(len(s)), key=lambda i: (-rem[i], i))
    for i in order[:short]:
        base[i] += 1
    return np.clip(np.array(base, dtype=np.int64), lo, hi).astype(np.int32)


def retained_layout(S: int, K_l) -> np.ndarray:
    """CSR offsets [H_kv + 1] of one batch element's retained entries.

    Head h's entries are rows out_off[h] .. out_off[h+1]-1 of the batch
    element's block; each head keeps min(K_l[h], S) entries.
    """
    kept = np.minimum(np.asarray(K_l, dtype=np.int64), S)
    return np.concatenate([[0], np.cumsum(kept)]).astype(np.int64)


def retained_cache_bytes(N: int, H_kv: int, K_l: int, D: int, B: int = 1,
                         elem_bytes: int = 2) -> int:
    """Bytes of the retained K and V over all layers (TideKV Fig. 5, Table 6)."""
    return N * B * H_kv * K_l * D * elem_bytes * 2
