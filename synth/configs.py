"""Workload shapes for layer-end compression (TideKV, Table 1 notation).

Symbols follow TideKV's notation table (Table 1): N layers, batch B, prompt
length S, prefill chunk C, H_q query heads, H_kv KV heads, head dim D.  The
scorer adds the observation window W, the key block b_s, the per-head budget
K_l and the mandatory sink/recent counts (TideKV, Fig. 3 caption), and the
pooling width.

The five shapes mirror the model layers the TideKV and HeteroCache pages
evaluate (Llama-3.1-8B, Mistral-7B, Qwen2.5-14B); nothing here is a model or
weights, only tensor shapes and the synthetic-input recipe.
"""

from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Config:
    name: str
    N: int            # layers in the model (TideKV, Table 1)
    B: int            # batch
    S: int            # prompt length
    C: int            # prefill chunk size (validated only; does not change the result)
    H_q: int
    H_kv: int
    D: int
    W: int            # observation window (last W prompt positions)
    b_s: int          # key block of the two-pass scan
    K_l: int          # per-head budget; 0 means "inverse-stability budgets"
    sink: int
    recent: int
    pool_k: int       # average-pool width (1 = no pooling)
    hh_frac: float    # fraction of positions made heavy hitters per (b, layer, KV head)
    seed: int
    budget_frac: float = 0.0   # total budget as a fraction of S * H_kv (inverse-stability mode)
    s_lo: float = 0.2          # stability scores drawn from U(s_lo, s_hi)
    s_hi: float = 1.0

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def GW(self) -> int:
        return self.G * self.W

    @property
    def inverse_stability(self) -> bool:
        return self.K_l == 0

    def with_(self, **kw) -> "Config":
        return replace(self, **kw)


CONFIGS = {
    # 1 layer, no pooling, recent = W as stated by the workload itself.
    "tiny": Config("tiny", N=1, B=1, S=512, C=512, H_q=4, H_kv=2, D=64, W=16,
                   b_s=128, K_l=128, sink=4, recent=16, pool_k=1, hh_frac=0.0,
                   seed=0),
    # Llama-3.1-8B layer shape at 8K.
    "llama8k": Config("llama8k", N=1, B=1, S=8192, C=2048, H_q=32, H_kv=8,
                      D=128, W=32, b_s=4096, K_l=1024, sink=4, recent=32,
                      pool_k=7, hh_frac=0.02, seed=1),
    # TideKV's main setting: 32 layers run layer-major, 64K, C=2048, budget 4096.
    "tidekv_main": Config("tidekv_main", N=32, B=1, S=65536, C=2048, H_q=32,
                          H_kv=8, D=128, W=32, b_s=4096, K_l=4096, sink=4,
                          recent=32, pool_k=7, hh_frac=0.02, seed=2),
    # Mistral-7B layer shape at 128K (32 layers in the model).
    "mistral128k": Config("mistral128k", N=32, B=1, S=131072, C=2048, H_q=32,
                          H_kv=8, D=128, W=64, b_s=4096, K_l=4096, sink=4,
                          recent=64, pool_k=7, hh_frac=0.03, seed=3),
    # Qwen2.5-14B layer shape, batch 4, 48 layers, per-KV-head budgets
    # proportional to 1/s with s ~ U(0.2, 1), 30% of S in total per layer.
    "qwen14b": Config("qwen14b", N=48, B=4, S=32768, C=2048, H_q=40, H_kv=8,
                      D=128, W=32, b_s=4096, K_l=0, sink=4, recent=32,
                      pool_k=7, hh_frac=0.02, seed=4, budget_frac=0.3),
}


def get_config(name: str, **overrides) -> Config:
    cfg = CONFIGS[name]
    return cfg.with_(**overrides) if overrides else cfg
