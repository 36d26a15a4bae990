"""CPU oracle for layer-major chunked prefill around the compress (test
infrastructure).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import this module.  It shares no code with the CUDA
library and imports nothing from it.

TideKV (Fig. 1(d), Fig. 2): the prompt streams chunk by chunk in layer-major
order; chunk j writes positions [j*C, min((j+1)*C, S)) of the active layer's
full KV; at the layer boundary the layer is compressed and its retained rows
and absolute positions are committed into the cross-layer cache C^[l]
(Fig. 4, cross-layer cache manager), after which the full KV is released.

Readings: a chunk tensor is [B, H_kv, c, D] with c = min(C, S - j*C); the
cross-layer cache stores the layers one after another, each laid out as
kvc_oracle.retained_layout describes for every batch element in turn.

Pins (tests/test_oracle_layer_major.py): chunks reassemble the prompt for
ragged and exact splits; the cache size at TideKV's main setting is the
512 MiB of its Fig. 5 / Tables 6 and 9; per-layer rows follow
kvc_oracle.retained_layout; budgets_pyramid matches hand-worked ramps (a
fractional one, a remainder tie) and stays within one key of the exact
rational ramp.
"""

from __future__ import annotations

import numpy as np

from . import kvc_oracle as O

__all__ = ["chunk_bounds", "assemble_chunks", "cache_layout", "compress_prefill", "budgets_pyramid"]


def chunk_bounds(S: int, C: int):
    """[(start, end)] of the prompt chunks."""
    return [(s, min(s + C, S)) for s in range(0, S, C)]


def assemble_chunks(chunks, S: int):
    """Active-layer buffer [B, H_kv, S, D] from the chunk tensors in order."""
    out = None
    pos = 0
    for c in chunks:
        c = np.asarray(c)
        if out is None:
            out = np.zeros(c.shape[:2] + (S,) + c.shape[3:], dtype=c.dtype)
        out[:, :, pos:pos + c.shape[2]] = c
        pos += c.shape[2]
    assert pos == S
    return out


def cache_layout(N: int, B: int, S: int, K_l) -> np.ndarray:
    """Row offsets [N + 1] of the layers in the cross-layer cache."""
    K_l = np.asarray(K_l).reshape(N, -1)
    out = np.zeros(N + 1, dtype=np.int64)
    for l in range(N):
        out[l + 1] = out[l] + B * int(O.retained_layout(S, K_l[l])[-1])
    return out


def compress_prefill(layers, K_l, sink: int, recent: int, pool_k: int):
    """Per layer, kvc_oracle.compress_layer of its full (assembled) KV."""
    return [O.compress_layer(q, k, v, K_l[l], sink, recent, pool_k) for l, (q, k, v) in enumerate(layers)]


def budgets_pyramid(N: int, budget: int, k_min: int) -> list:
    """Per-layer budgets shrinking linearly from 2*budget - k_min to k_min.

    TideKV's Tables 3-4 run a PyramidKV selector at a given average budget;
    the pages give no schedule.  Reading: a linear ramp with mean = budget,
    exact shares rounded by largest remainder (ties to the lower layer) so
    that the layers sum to N * budget.  Parity unpinned beyond that sum, the
    ramp's ends and its monotonicity.
    """
    if N == 1:
        return [budget]
    k_max = 2.0 * budget - k_min
    exact = [k_max - (k_max - k_min) * l / (N - 1) for l in range(N)]
    base = [int(np.floor(x)) for x in exact]
    short = N * budget - sum(base)
    rem = [x - b for x, b in zip(exact, base)]
    for i in sorted(range(N), key=lambda i: (-rem[i], i))[:short]:
        base[i] += 1
    return base
