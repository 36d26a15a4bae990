"""Shared helpers of the GPU parity tests: run the CUDA path through the
C ABI, and compare its outputs with the oracle's under the stated tolerances.

Tolerances (bf16 inputs, fp32 accumulation):
  m:       |gpu - oracle| <= 2e-3 * max(1, |m|)
  Z:       |gpu - oracle| <= 2e-3 * Z
  scores:  |gpu - oracle| <= 2e-3 * |oracle| + 2e-3 * (G*W / S)   (the second
           term is 2e-3 of the mean per-key mass, since sum_j r_j = G*W)
  selection: with theta the n_sel-th largest oracle score among the
           non-mandatory keys, keys scoring above theta*(1+2e-3) must be kept
           and keys below theta*(1-2e-3) dropped; inside that band any choice
           of the right size is valid.  R_mand is always kept and every head
           keeps exactly min(K_l, S) keys in ascending order.
  gather:  bit-exact against the oracle's gather at the GPU's own indices.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import kvc_oracle as O

TOL = 2e-3


def kl_vector(cfg, K, layer=0):
    """(K_l for the CUDA side, K_l for the oracle side) of one layer."""
    if not cfg.inverse_stability:
        v = [cfg.K_l] * cfg.H_kv
        return v, list(v)
    from synth import stability_scores
    s = stability_scores(cfg, layer).numpy()
    total = round(cfg.budget_frac * cfg.S * cfg.H_kv)
    rsz = len(O.mandatory_set(cfg.S, cfg.sink, cfg.recent))
    gpu = K.kvc_budget_inverse_stability(s, total, rsz, cfg.S)
    ref = O.budgets_inverse_stability(s, total, rsz, cfg.S).tolist()
    assert gpu == ref
    return gpu, ref


def to_dev(inp, dev="cuda"):
    return inp.q_win.to(dev), inp.k.to(dev), inp.v.to(dev)


def run_compress(K, cfg, inp, K_l, layer=0, ws=None, dev="cuda"):
    q, k, v = to_dev(inp, dev)
    k_out, v_out, pos, off = K.retained_outputs(cfg.B, cfg.H_kv, cfg.S, cfg.D, K_l, device=dev)
    if ws is None:
        ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, max(K_l), cfg.pool_k, device=dev)
    K.kvc_compress_layer(cfg.N, layer, cfg.B, cfg.S, cfg.C, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, K_l, cfg.sink,
                         cfg.recent, cfg.pool_k, cfg.b_s, q, k, v, k_out, v_out, pos, ws)
    K.kvc_check_status()
    return k_out.cpu(), v_out.cpu(), pos.cpu(), off


def run_decomposed(K, cfg, inp, K_l, dev="cuda"):
    q, k, v = to_dev(inp, dev)
    B, Hq, Hkv, S, D, W = cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W
    ws = K.workspace(B, Hq, Hkv, D, W, cfg.b_s, max(K_l), cfg.pool_k, device=dev)
    m = torch.empty((B, Hq, W), dtype=torch.float32, device=dev)
    Z = torch.empty_like(m)
    K.kvc_score_pass1(q, k, B, Hq, Hkv, S, D, W, cfg.b_s, m, Z, ws)
    scores = torch.empty((B, Hkv, S), dtype=torch.float32, device=dev)
    K.kvc_score_pass2_pool(q, k, m, Z, B, Hq, Hkv, S, D, W, cfg.b_s, cfg.pool_k, scores, ws)
    k_out, v_out, pos, off = K.retained_outputs(B, Hkv, S, D, K_l, device=dev)
    idx = torch.empty_like(pos)
    K.kvc_select_topk(scores, B, Hkv, S, K_l, cfg.sink, cfg.recent, idx, ws)
    K.kvc_gather(k, v, idx, B, Hkv, S, D, K_l, k_out, v_out, pos)
    K.kvc_check_status()
    return dict(m=m.cpu(), Z=Z.cpu(), scores=scores.cpu(), idx=idx.cpu(), k_out=k_out.cpu(),
                v_out=v_out.cpu(), pos=pos.cpu(), off=off)


def oracle_head(cfg, inp, b, h):
    G = cfg.H_q // cfg.H_kv
    q = O.as_f64(inp.q_win[b, h * G:(h + 1) * G]).reshape(G * cfg.W, cfg.D)
    return O.score_head(q, inp.k[b, h], cfg.W, cfg.pool_k)


def assert_scores_close(gpu, ref, cfg, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    floor = TOL * (cfg.G * cfg.W) / cfg.S
    err = np.abs(gpu - ref)
    bad = err > TOL * np.abs(ref) + floor
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at "
                           f"{int(np.argmax(err - TOL * np.abs(ref)))}: gpu={gpu.ravel()[np.argmax(err - TOL*np.abs(ref))]}"
                           f" ref={ref.ravel()[np.argmax(err - TOL*np.abs(ref))]}")


def assert_mz_close(m_gpu, Z_gpu, o, what):
    m_gpu = np.asarray(m_gpu, dtype=np.float64)
    Z_gpu = np.asarray(Z_gpu, dtype=np.float64)
    assert np.all(np.abs(m_gpu - o["m"]) <= TOL * np.maximum(1.0, np.abs(o["m"]))), f"{what}: m"
    assert np.all(np.abs(Z_gpu - o["Z"]) <= TOL * o["Z"]), f"{what}: Z"


def check_selection(idx, s_ref, K_l, cfg, what):
    """Selection of one head against oracle scores with the tie band."""
    S = cfg.S
    idx = np.asarray(idx, dtype=np.int64)
    kept = min(K_l, S)
    assert len(idx) == kept, f"{what}: {len(idx)} kept, expected {kept}"
    assert np.all(np.diff(idx) > 0), f"{what}: not strictly ascending"
    assert idx.min() >= 0 and idx.max() < S
    R = O.mandatory_set(S, cfg.sink, cfg.recent)
    chosen = set(idx.tolist())
    assert set(R.tolist()) <= chosen, f"{what}: mandatory key dropped"
    if K_l >= S:
        return
    n_sel = K_l - len(R)
    mask = np.ones(S, dtype=bool)
    mask[R] = False
    cand = np.nonzero(mask)[0]
    if n_sel == 0:
        assert chosen == set(R.tolist())
        return
    order = np.lexsort((cand, -s_ref[cand]))
    theta = s_ref[cand[order[n_sel - 1]]]
    hi = cand[s_ref[cand] > theta * (1 + TOL)]
    lo = cand[s_ref[cand] < theta * (1 - TOL)]
    missing = set(hi.tolist()) - chosen
    extra = set(lo.tolist()) & chosen
    assert not missing, f"{what}: {len(missing)} keys above the tie band dropped, e.g. {sorted(missing)[:5]}"
    assert not extra, f"{what}: {len(extra)} keys below the tie band kept, e.g. {sorted(extra)[:5]}"


def check_head_outputs(k_out, v_out, pos, off, inp, cfg, b, h, K_l_h, s_ref, what):
    T = off[-1]
    lo, hi = b * T + off[h], b * T + off[h + 1]
    idx = pos[lo:hi].numpy().astype(np.int64)
    check_selection(idx, s_ref, K_l_h, cfg, what)
    kh, vh, p = O.gather(inp.k[b, h], inp.v[b, h], idx)
    assert torch.equal(k_out[lo:hi].view(torch.int16), kh.view(torch.int16)), f"{what}: K gather"
    assert torch.equal(v_out[lo:hi].view(torch.int16), vh.view(torch.int16)), f"{what}: V gather"
    assert np.array_equal(pos[lo:hi].numpy(), p), f"{what}: positions"


def check_structure_all_heads(pos, off, cfg, K_l):
    """Properties that hold for every head at any size."""
    T = off[-1]
    R = set(O.mandatory_set(cfg.S, cfg.sink, cfg.recent).tolist())
    P = pos.numpy()
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            seg = P[b * T + off[h]: b * T + off[h + 1]]
            assert len(seg) == min(K_l[h], cfg.S)
            assert np.all(np.diff(seg) > 0) and seg[0] >= 0 and seg[-1] < cfg.S
            assert R <= set(seg.tolist())
