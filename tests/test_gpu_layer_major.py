"""GPU parity of layer-major chunked prefill around the compress (TideKV,
Fig. 1(d), Fig. 2): chunks appended into the active layer's buffer must
rebuild the prompt's keys and values bit for bit, and each layer compressed
straight into its rows of the cross-layer cache must match the oracle
(selection within the tie band, gather bit-exact, positions = indices)."""

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from oracle import layer_major as LM
from synth import get_config, make_layer_inputs
from tests import kvc_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import attention_score_kv_gb300.kvc as K
    return K


@pytest.mark.parametrize("D,C", [(128, 128), (64, 96)])
def test_prefill_three_layers_into_the_cross_layer_cache(K, D, C):
    cfg = get_config("tiny", N=3, S=700, C=C, H_q=8, H_kv=2, D=D, W=16, K_l=200, recent=16, pool_k=7,
                     hh_frac=0.02, seed=41)
    _prefill_and_check(K, cfg, [[200, 260], [200, 150], [700, 40]])   # unequal heads and layers, one keeps all


def test_prefill_with_pyramid_budgets(K):
    """Per-layer budgets from the PyramidKV-style ramp (TideKV-PyramidKV,
    Tables 3-4) drive the compress of four layers."""
    cfg = get_config("tiny", N=4, S=900, C=256, H_q=8, H_kv=2, D=128, W=16, K_l=200, recent=16, pool_k=7,
                     hh_frac=0.02, seed=43)
    pyr = K.kvc_budget_pyramid(cfg.N, 200, 40)
    assert pyr == [int(x) for x in LM.budgets_pyramid(cfg.N, 200, 40)]
    assert sum(pyr) == cfg.N * 200 and pyr == sorted(pyr, reverse=True) and pyr[-1] == 40
    _prefill_and_check(K, cfg, [[k] * cfg.H_kv for k in pyr])


def _prefill_and_check(K, cfg, K_l):
    dev = "cuda"
    off_layers = K.kvc_cache_layout(cfg.N, cfg.B, cfg.H_kv, cfg.S, K_l)
    assert off_layers == LM.cache_layout(cfg.N, cfg.B, cfg.S, K_l).tolist()
    rows = off_layers[-1]
    cache_k = torch.empty((rows, cfg.D), dtype=torch.bfloat16, device=dev)
    cache_v = torch.empty_like(cache_k)
    cache_p = torch.empty((rows,), dtype=torch.int32, device=dev)
    k_act = torch.full((cfg.B, cfg.H_kv, cfg.S, cfg.D), 7.0, dtype=torch.bfloat16, device=dev)
    v_act = torch.full_like(k_act, -3.0)
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, 700, cfg.pool_k, device=dev)
    layers = []
    for l in range(cfg.N):
        inp = make_layer_inputs(cfg, l)
        layers.append(inp)
        for j, (a, b) in enumerate(LM.chunk_bounds(cfg.S, cfg.C)):
            kc = inp.k[:, :, a:b].contiguous().to(dev)
            vc = inp.v[:, :, a:b].contiguous().to(dev)
            K.kvc_append_chunk(kc, vc, cfg.B, cfg.H_kv, cfg.S, cfg.C, cfg.D, j, k_act, v_act)
        assert torch.equal(k_act.cpu().view(torch.int16), inp.k.view(torch.int16)), f"layer {l}: K buffer"
        assert torch.equal(v_act.cpu().view(torch.int16), inp.v.view(torch.int16)), f"layer {l}: V buffer"
        lo, hi = off_layers[l], off_layers[l + 1]
        K.kvc_compress_layer(cfg.N, l, cfg.B, cfg.S, cfg.C, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, K_l[l], cfg.sink,
                             cfg.recent, cfg.pool_k, cfg.b_s, inp.q_win.to(dev), k_act, v_act, cache_k[lo:hi],
                             cache_v[lo:hi], cache_p[lo:hi], ws)
    K.kvc_check_status()
    ck, cv, cp = cache_k.cpu(), cache_v.cpu(), cache_p.cpu()
    for l, inp in enumerate(layers):
        lo, hi = off_layers[l], off_layers[l + 1]
        off = O.retained_layout(cfg.S, K_l[l])
        for b in range(cfg.B):
            for h in range(cfg.H_kv):
                o = U.oracle_head(cfg, inp, b, h)
                U.check_head_outputs(ck[lo:hi], cv[lo:hi], cp[lo:hi], off, inp, cfg, b, h, K_l[l][h], o["s"],
                                     f"layer {l} b={b} h={h}")


def test_chunk_beyond_the_prompt_is_rejected(K):
    k = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16, device="cuda")
    act = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(K.KvcError) as e:
        K.kvc_append_chunk(k, k, 1, 1, 16, 8, 64, 2, act, act)
    assert e.value.code == -1
