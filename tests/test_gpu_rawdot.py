"""GPU parity of the single-pass INT8 raw inner-product scorer (HillInfer).

Every step of the scorer is one correctly rounded float32 operation or exact
integer arithmetic, so the scores must equal the oracle's bit for bit; the
selection then decides on identical numbers and must agree exactly, and the
gather is a bit copy.  Runs through the C ABI.
"""

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from oracle import rawdot_int8 as R
from synth import get_config, make_layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import attention_score_kv_gb300.kvc as K
    return K


SHAPES = {
    "tiny": dict(base="tiny"),
    "d64_ragged": dict(base="tiny", S=777, C=777, H_q=6, H_kv=2, D=64, W=5, K_l=100, recent=5, sink=2, seed=31),
    "d128_gw256": dict(base="tiny", S=1500, C=1500, H_q=8, H_kv=1, D=128, W=32, K_l=400, recent=32, seed=32,
                       hh_frac=0.02),
    "b2_gw160": dict(base="tiny", B=2, S=2100, C=2100, H_q=10, H_kv=2, D=128, W=32, K_l=600, recent=32, seed=33),
    "s_one": dict(base="tiny", S=1, C=1, W=1, sink=0, recent=1, K_l=1, seed=34),
}


def _cfg(name):
    d = dict(SHAPES[name])
    return get_config(d.pop("base"), **d)


def _run_scores(K, cfg, q, k):
    dev = "cuda"
    scores = torch.empty((cfg.B, cfg.H_kv, cfg.S), dtype=torch.float32, device=dev)
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, cfg.K_l, cfg.pool_k, device=dev)
    K.kvc_score_rawdot_int8(q.to(dev), k.to(dev), cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W, scores, ws)
    K.kvc_check_status()
    return scores.cpu().numpy(), ws


def _bits(x):
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_scores_bit_exact_and_selection_exact(K, name):
    cfg = _cfg(name)
    inp = make_layer_inputs(cfg)
    got, ws = _run_scores(K, cfg, inp.q_win, inp.k)
    G = cfg.G
    K_l = [min(cfg.K_l, cfg.S)] * cfg.H_kv
    idx = torch.empty((cfg.B, sum(K_l)), dtype=torch.int32, device="cuda")
    K.kvc_select_topk(torch.from_numpy(got).cuda(), cfg.B, cfg.H_kv, cfg.S, K_l, cfg.sink, cfg.recent, idx, ws)
    K.kvc_check_status()
    idx = idx.cpu().numpy()
    off = np.concatenate([[0], np.cumsum(K_l)])
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            qg = inp.q_win[b, h * G:(h + 1) * G].reshape(G * cfg.W, cfg.D)
            ref = R.raw_scores_int8_rows(qg, inp.k[b, h])
            assert np.array_equal(_bits(got[b, h]), _bits(ref)), f"{name} b={b} h={h}"
            sel = O.select_topk(ref.astype(np.float64), K_l[h], cfg.sink, cfg.recent)
            assert idx[b, off[h]:off[h + 1]].tolist() == sel.tolist(), f"{name} b={b} h={h}"


def test_zero_rows_and_zero_query_score_zero(K):
    cfg = _cfg("tiny")
    inp = make_layer_inputs(cfg)
    k = inp.k.clone()
    k[0, 0, 5] = 0
    k[0, 1, 17] = 0
    got, _ = _run_scores(K, cfg, inp.q_win, k)
    assert got[0, 0, 5] == 0 and got[0, 1, 17] == 0
    got, _ = _run_scores(K, cfg, torch.zeros_like(inp.q_win), inp.k)
    assert not np.any(got)


def test_selection_of_signed_dense_scores_is_exact(K):
    rng = np.random.default_rng(5)
    B, H, S = 2, 3, 5000
    s = rng.standard_normal((B, H, S)).astype(np.float32)
    s[0, 0, ::7] = -1.5                        # many exact ties, negative
    s[1, 2, 100:4000] = 0.0                    # a long run of equal zeros ...
    s[1, 2, 200:300] = -0.0                    # ... some of them negative zero
    K_l = [1000, 37, 4999]
    sink, recent = 3, 9
    idx = torch.empty((B, sum(K_l)), dtype=torch.int32, device="cuda")
    ws = K.workspace(B, H, H, 64, 1, 128, max(K_l), 1, device="cuda")
    K.kvc_select_topk(torch.from_numpy(s).cuda(), B, H, S, K_l, sink, recent, idx, ws)
    K.kvc_check_status()
    idx = idx.cpu().numpy()
    off = np.concatenate([[0], np.cumsum(K_l)])
    for b in range(B):
        for h in range(H):
            ref = O.select_topk(s[b, h].astype(np.float64), K_l[h], sink, recent)
            assert idx[b, off[h]:off[h + 1]].tolist() == ref.tolist(), (b, h)


def test_full_size_mistral_sampled_heads(K):
    cfg = get_config("mistral128k")
    inp = make_layer_inputs(cfg, 0, device="cuda")
    scores = torch.empty((cfg.B, cfg.H_kv, cfg.S), dtype=torch.float32, device="cuda")
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, cfg.K_l, cfg.pool_k, device="cuda")
    K.kvc_score_rawdot_int8(inp.q_win, inp.k, cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W, scores, ws)
    K.kvc_check_status()
    G = cfg.G
    for h in (0, cfg.H_kv - 1):
        qg = inp.q_win[0, h * G:(h + 1) * G].reshape(G * cfg.W, cfg.D).cpu()
        ref = R.raw_scores_int8_rows(qg, inp.k[0, h].cpu())
        assert np.array_equal(_bits(scores[0, h].cpu().numpy()), _bits(ref)), f"head {h}"
