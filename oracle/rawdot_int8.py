"""CPU oracle for the single-pass raw inner-product scorer with INT8 keys.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import this module.  It shares no code with the CUDA
library and imports nothing from it.

HillInfer ("Algorithmic Simplification"): because the softmax is strictly
monotone and eviction only ranks tokens, the scorer drops the exponentials
and the 1/sqrt(d) scaling and ranks by the raw inner product Q.K^T.
HillInfer ("Streaming Execution and Asymmetric Precision"): the inner
products run in low precision (INT8) on keys cast on the fly from the
stored 16-bit values; the kept tokens are then fetched at full precision.

Readings taken where the page leaves a step open:
  * one scoring query per KV head: the sum of the group's G*W window queries.
    Raw inner products are linear, so q_bar . k_j equals the window-and-group
    sum of q_{g,i} . k_j, i.e. the two-pass score with the softmax removed
    (and without the causal mask, which only touches recent keys, all of
    them mandatory);
  * q_bar is summed in float32, row by row in (g, i) order;
  * symmetric per-row INT8: amax = max |x|, code = rint(x * (127 / amax))
    clamped to [-127, 127] (round half to even), scale = amax / 127, all in
    float32; an all-zero row has codes 0 and scale 0;
  * score_j = float32(float32(dot_j) * scale_q) * scale_k, with dot_j the
    exact integer sum of code products;
  * no pooling.

Functions and their pins (tests/test_oracle_rawdot.py):
  summed_query: the fp64 window/group sum of raw logits (through
      kvc_oracle.dense_logits) outside the causal band.
  quantize_int8: a hand-worked example, a hand-worked row of exact .5 ties
      (round half to even), extremes at +-127, zero rows, and the rounding
      error bound.
  raw_scores_exact / raw_scores_int8: the analytic quantisation error bound;
      for one query (G = W = 1) the exact raw ranking equals the softmax
      oracle's selection (HillInfer's monotonicity argument).
"""

from __future__ import annotations

import numpy as np

__all__ = ["summed_query", "quantize_int8", "raw_scores_exact", "raw_scores_int8", "raw_scores_int8_rows",
           "int8_error_bound"]

_F127 = np.float32(127.0)


def _f32(x) -> np.ndarray:
    """bf16 (torch) or any array -> float32 numpy, exactly."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float32)


def summed_query(q_grp) -> np.ndarray:
    """q_bar[d] = sum over the rows of q_grp [G*W, D], in float32, row order."""
    q = _f32(q_grp)
    acc = np.zeros(q.shape[1], dtype=np.float32)
    for r in range(q.shape[0]):
        acc = (acc + q[r]).astype(np.float32)
    return acc


def quantize_int8(x) -> tuple[np.ndarray, np.float32]:
    """Symmetric INT8 codes of one float32 row and its scale (see header)."""
    x = _f32(x)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    if amax == 0:
        return np.zeros(x.shape, dtype=np.int32), np.float32(0.0)
    inv = np.float32(_F127 / amax)
    codes = np.rint((x * inv).astype(np.float32)).astype(np.int32)
    codes = np.clip(codes, -127, 127)
    return codes, np.float32(amax / _F127)


def raw_scores_exact(q_grp, k) -> np.ndarray:
    """fp64 q_bar . k_j for every key j (q_bar summed in fp64)."""
    q = _f32(q_grp).astype(np.float64)
    kk = _f32(k).astype(np.float64)
    return kk @ q.sum(axis=0)


def raw_scores_int8(q_grp, k) -> np.ndarray:
    """float32 INT8 raw scores of every key of one head (see header), one key
    at a time."""
    qc, sq = quantize_int8(summed_query(q_grp))
    kk = _f32(k)
    out = np.empty(kk.shape[0], dtype=np.float32)
    for j in range(kk.shape[0]):
        kc, sk = quantize_int8(kk[j])
        dot = int(np.dot(qc.astype(np.int64), kc.astype(np.int64)))
        out[j] = np.float32(np.float32(np.float32(dot) * sq) * sk)
    return out


def raw_scores_int8_rows(q_grp, k) -> np.ndarray:
    """raw_scores_int8 for many keys at once: the same float32 operations,
    element by element, on whole arrays (for full-size heads)."""
    qc, sq = quantize_int8(summed_query(q_grp))
    kk = _f32(k)
    amax = np.max(np.abs(kk), axis=1).astype(np.float32)
    nz = amax > 0
    inv = np.zeros_like(amax)
    inv[nz] = (_F127 / amax[nz]).astype(np.float32)
    codes = np.clip(np.rint((kk * inv[:, None]).astype(np.float32)), -127, 127).astype(np.int64)
    codes[~nz] = 0
    sk = np.zeros_like(amax)
    sk[nz] = (amax[nz] / _F127).astype(np.float32)
    dot = codes @ qc.astype(np.int64)
    return ((dot.astype(np.float32) * sq).astype(np.float32) * sk).astype(np.float32)


def int8_error_bound(q_grp, k) -> np.ndarray:
    """Bound on |raw_scores_int8 - q_bar32 . k_j| from code rounding.

    With x = s*c + e, |e| <= s/2 per element (the clamp never binds because
    the largest element maps to exactly 127):
    |q.k - s_q s_k c_q.c_k| <= sum_d (|q_d| s_k/2 + |k_d| s_q/2 + s_q s_k/4),
    plus a few float32 roundings of the product, allowed for by a relative
    2^-20 of sum_d |q_d k_d|.
    """
    qb = summed_query(q_grp).astype(np.float64)
    _, sq = quantize_int8(qb.astype(np.float32))
    kk = _f32(k).astype(np.float64)
    bound = np.empty(kk.shape[0])
    for j in range(kk.shape[0]):
        _, sk = quantize_int8(kk[j].astype(np.float32))
        bound[j] = (np.abs(qb).sum() * float(sk) / 2 + np.abs(kk[j]).sum() * float(sq) / 2
                    + kk.shape[1] * float(sq) * float(sk) / 4 + 2.0 ** -20 * np.abs(qb * kk[j]).sum())
    return bound
