"""Seeded synthetic Q/K/V for one layer, plus seeded head-stability draws.

Recipe (one layer l of workload ``cfg``):

* A ``torch.Generator`` on ``device`` is seeded with ``cfg.seed * 1000 + l``.
* Q_win ``[B, H_q, W, D]``, K and V ``[B, H_kv, S, D]`` are drawn N(0, 1) in
  fp32, in that order.
* Heavy hitters: for every (b, KV head h), ``ceil(hh_frac * S)`` positions are
  drawn uniformly without replacement (``randperm``).  Their keys get
  ``c * u`` added, where ``u`` is the unit vector along the mean of the head's
  G*W window queries and ``c = heavy_hitter_scale(D)``.
* Q, K, V are then rounded to bf16.  The same bf16 bytes feed the oracle
  and the CUDA path.

Nothing here computes any part of the compression method.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

from .configs import Config


def heavy_hitter_scale(D: int, c: float | None = None) -> float:
    """Magnitude of the query-aligned shift given to heavy-hitter keys.

    "+3 * unit" taken literally would move a logit by only 3/sqrt(D) (about
    0.27 at D=128), which does not make a key heavy; the default reads it as a
    shift of about +3 in logit units, i.e. ``3 * sqrt(D)`` along the unit
    vector.  Pass ``c`` to use another magnitude.
    """
    return 3.0 * math.sqrt(D) if c is None else float(c)


@dataclass
class LayerInputs:
    q_win: torch.Tensor   # [B, H_q, W, D] bf16
    k: torch.Tensor       # [B, H_kv, S, D] bf16
    v: torch.Tensor       # [B, H_kv, S, D] bf16
    hh_pos: torch.Tensor  # [B, H_kv, n_hh] int64 heavy-hitter positions (may be empty)


def make_layer_inputs(cfg: Config, layer: int = 0, device: str | torch.device = "cpu",
                      hh_c: float | None = None, seed: int | None = None) -> LayerInputs:
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed((cfg.seed if seed is None else seed) * 1000 + layer)
    B, Hq, Hkv, S, D, W = cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W
    G = Hq // Hkv
    q = torch.randn((B, Hq, W, D), generator=gen, device=dev, dtype=torch.float32)
    k = torch.randn((B, Hkv, S, D), generator=gen, device=dev, dtype=torch.float32)
    v = torch.randn((B, Hkv, S, D), generator=gen, device=dev, dtype=torch.float32)
    n_hh = math.ceil(cfg.hh_frac * S) if cfg.hh_frac > 0 else 0
    hh = torch.empty((B, Hkv, n_hh), dtype=torch.int64, device=dev)
    if n_hh:
        c = heavy_hitter_scale(D, hh_c)
        qg = q.view(B, Hkv, G * W, D)
        for b in range(B):
            for h in range(Hkv):
                pos = torch.randperm(S, generator=gen, device=dev)[:n_hh]
                u = qg[b, h].mean(dim=0)
                u = u / u.norm()
                k[b, h, pos] += c * u
                hh[b, h] = pos
    return LayerInputs(q.to(torch.bfloat16), k.to(torch.bfloat16),
                       v.to(torch.bfloat16), hh)


def stability_scores(cfg: Config, layer: int = 0) -> torch.Tensor:
    """Per-KV-head stability scores s ~ U(s_lo, s_hi), float64, shape [H_kv].

    Drawn from their own CPU generator (seed ``cfg.seed * 1000 + 500 + layer``)
    so they do not depend on the device the tensors were drawn on.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(cfg.seed * 1000 + 500 + layer)
    u = torch.rand((cfg.H_kv,), generator=gen, dtype=torch.float64)
    return cfg.s_lo + (cfg.s_hi - cfg.s_lo) * u
