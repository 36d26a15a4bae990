"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small shapes (several 128-key tiles, ragged tails, edge cases) are compared
element by element on every head; the five workload shapes at full size are
compared on sampled heads (the oracle materialises one head's dense softmax at
a time) plus structural properties on every head.
"""

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from synth import get_config, make_layer_inputs
from tests import kvc_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_score_kv_gb300 import build
    build.build()
    import attention_score_kv_gb300.kvc as kvc
    return kvc


SMALL = {
    "tiny": dict(base="tiny"),
    "tiny_pool7": dict(base="tiny", pool_k=7),
    "ragged_S1000": dict(base="tiny", S=1000, C=1000, H_q=8, H_kv=2, D=128, W=32, pool_k=7, K_l=300,
                         recent=32, hh_frac=0.02, seed=11),
    "odd_gw15_d64": dict(base="tiny", S=777, C=777, H_q=6, H_kv=2, D=64, W=5, pool_k=5, K_l=100,
                         recent=5, sink=2, hh_frac=0.03, seed=12),
    "gw256_max": dict(base="tiny", S=1500, C=1500, H_q=8, H_kv=1, D=128, W=32, pool_k=7, K_l=400,
                      recent=32, hh_frac=0.02, seed=13),
    "gw160_qwen_like": dict(base="tiny", S=2100, C=2100, H_q=10, H_kv=2, D=128, W=32, pool_k=7, K_l=600,
                            recent=32, hh_frac=0.02, seed=14, B=2),
    "w_equals_s": dict(base="tiny", S=64, C=64, W=64, recent=64, sink=0, K_l=64, seed=15),
    "k_ge_s": dict(base="tiny", S=300, C=300, K_l=1000, seed=16),
    "k_eq_mandatory": dict(base="tiny", S=400, C=400, K_l=20, seed=17),
    "sink_recent_overlap": dict(base="tiny", S=40, C=40, W=16, sink=30, recent=20, K_l=40, seed=18),
    "s_one": dict(base="tiny", S=1, C=1, W=1, sink=0, recent=1, K_l=1, seed=19),
    "pool15": dict(base="tiny", S=900, C=900, pool_k=15, sink=8, K_l=200, seed=20),
    "b3_no_sink": dict(base="tiny", B=3, S=640, C=640, sink=0, recent=16, K_l=100, seed=21, hh_frac=0.05),
}


def small_cfg(name):
    d = dict(SMALL[name])
    return get_config(d.pop("base"), **d)


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_decomposed_every_head(K, name):
    cfg = small_cfg(name)
    inp = make_layer_inputs(cfg)
    K_l, K_l_ref = U.kl_vector(cfg, K)
    out = U.run_decomposed(K, cfg, inp, K_l)
    G = cfg.G
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            o = U.oracle_head(cfg, inp, b, h)
            U.assert_mz_close(out["m"][b, h * G:(h + 1) * G].reshape(-1), out["Z"][b, h * G:(h + 1) * G].reshape(-1),
                              o, f"{name} b={b} h={h}")
            U.assert_scores_close(out["scores"][b, h].numpy(), o["s"], cfg, f"{name} scores b={b} h={h}")
            U.check_head_outputs(out["k_out"], out["v_out"], out["pos"], out["off"], inp, cfg, b, h,
                                 K_l_ref[h], o["s"], f"{name} decomposed b={b} h={h}")


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_compress_layer_every_head(K, name):
    cfg = small_cfg(name)
    inp = make_layer_inputs(cfg)
    K_l, K_l_ref = U.kl_vector(cfg, K)
    k_out, v_out, pos, off = U.run_compress(K, cfg, inp, K_l)
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            o = U.oracle_head(cfg, inp, b, h)
            U.check_head_outputs(k_out, v_out, pos, off, inp, cfg, b, h, K_l_ref[h], o["s"],
                                 f"{name} compress b={b} h={h}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 5])
def test_candidate_compaction_path(K, ctas):
    """Few scan CTAs: each key range sees far more keys than its candidate
    capacity (K_l_max + b_s), so the in-kernel compaction runs; with an odd
    CTA count the ranges also straddle the two heads."""
    cfg = get_config("tiny", S=6000, C=6000, H_q=8, H_kv=2, D=128, W=32, pool_k=7, K_l=200, recent=32,
                     b_s=128, hh_frac=0.02, seed=30 + ctas)
    inp = make_layer_inputs(cfg)
    K_l, K_l_ref = U.kl_vector(cfg, K)
    K.kvc_set_option(K.KVC_OPT_SCAN_CTAS, ctas)
    try:
        k_out, v_out, pos, off = U.run_compress(K, cfg, inp, K_l)
    finally:
        K.kvc_set_option(K.KVC_OPT_SCAN_CTAS, 0)
    for h in range(cfg.H_kv):
        o = U.oracle_head(cfg, inp, 0, h)
        U.check_head_outputs(k_out, v_out, pos, off, inp, cfg, 0, h, K_l_ref[h], o["s"], f"compaction ctas={ctas} h={h}")


# (H_kv, S, scan CTAs) whose key-range boundaries land near head boundaries:
# one snapped back onto a head start; one 76 keys past the snap distance (a
# real two-segment CTA); one snapped forward at 232 keys next to a 234-key
# near miss (the distance is 233); one forward and one back, both exactly at
# the distance (140).
SNAP_CASES = [(2, 700, 6), (2, 700, 9), (4, 700, 3), (4, 700, 5)]


@pytest.mark.parametrize("H_kv,S,ctas", SNAP_CASES)
def test_range_snapping_every_head(K, H_kv, S, ctas):
    """Forced scan-CTA counts put range boundaries at and around the snap
    distance from head boundaries; the compress path and the decomposed path
    (whose pass-1 partials are merged per head by range) must both match the
    oracle on every head."""
    cfg = get_config("tiny", S=S, C=S, H_q=2 * H_kv, H_kv=H_kv, D=64, W=16, pool_k=5, K_l=150, recent=16,
                     hh_frac=0.03, seed=50 + ctas)
    inp = make_layer_inputs(cfg)
    K_l, K_l_ref = U.kl_vector(cfg, K)
    K.kvc_set_option(K.KVC_OPT_SCAN_CTAS, ctas)
    try:
        k_out, v_out, pos, off = U.run_compress(K, cfg, inp, K_l)
        dec = U.run_decomposed(K, cfg, inp, K_l)
    finally:
        K.kvc_set_option(K.KVC_OPT_SCAN_CTAS, 0)
    G = cfg.G
    for h in range(cfg.H_kv):
        o = U.oracle_head(cfg, inp, 0, h)
        what = f"H_kv={H_kv} S={S} ctas={ctas} h={h}"
        U.check_head_outputs(k_out, v_out, pos, off, inp, cfg, 0, h, K_l_ref[h], o["s"], what + " compress")
        U.assert_mz_close(dec["m"][0, h * G:(h + 1) * G].reshape(-1), dec["Z"][0, h * G:(h + 1) * G].reshape(-1),
                          o, what + " pass 1")
        U.assert_scores_close(dec["scores"][0, h].numpy(), o["s"], cfg, what + " scores")


def _select_case(K, S, H_kv, B, K_l, sink, recent, scores64):
    """GPU selection on given fp32 scores must equal the oracle's selection on
    the same fp32 values exactly (both decide in fp32)."""
    s32 = torch.from_numpy(scores64.astype(np.float32))
    cfg_ws = K.workspace(B, H_kv, H_kv, 64, 1, 128, max(K_l), 1)
    off = K.kvc_retained_layout(H_kv, S, K_l)
    idx = torch.empty((B * off[-1],), dtype=torch.int32, device="cuda")
    K.kvc_select_topk(s32.cuda(), B, H_kv, S, K_l, sink, recent, idx, cfg_ws)
    K.kvc_check_status()
    idx = idx.cpu().numpy()
    for b in range(B):
        for h in range(H_kv):
            ref = O.select_topk(s32[b, h].double().numpy(), K_l[h], sink, recent)
            got = idx[b * off[-1] + off[h]: b * off[-1] + off[h + 1]]
            assert np.array_equal(got, ref), f"b={b} h={h}"


def test_select_exact_random_scores(K):
    rng = np.random.default_rng(1)
    B, H, S = 2, 3, 5000
    _select_case(K, S, H, B, [100, 777, 2500], 4, 32, rng.random((B, H, S)))


def test_select_exact_many_ties(K):
    rng = np.random.default_rng(2)
    B, H, S = 1, 4, 4096
    s = np.round(rng.random((B, H, S)) * 20) / 20          # 21 distinct values
    _select_case(K, S, H, B, [50, 500, 1000, 4000], 4, 16, s)


def test_select_exact_all_equal_and_edges(K):
    S = 3000
    s = np.full((1, 4, S), 0.25)
    s[0, 1, 100:200] = 0.0                                    # zeros
    _select_case(K, S, 4, 1, [20, 3000, 20 + 1, 5000], 4, 16, s)


def test_select_exact_oracle_scores(K):
    cfg = get_config("llama8k")
    inp = make_layer_inputs(cfg)
    s = np.stack([[U.oracle_head(cfg, inp, 0, h)["s"] for h in range(2)]])
    _select_case(K, cfg.S, 2, 1, [cfg.K_l, 2 * cfg.K_l], cfg.sink, cfg.recent, s)


def test_gather_bit_exact(K):
    cfg = get_config("tiny", S=2000, C=2000, D=128)
    inp = make_layer_inputs(cfg)
    rng = np.random.default_rng(3)
    K_l = [300, 77]
    off = K.kvc_retained_layout(2, cfg.S, K_l)
    idx = np.concatenate([np.sort(rng.choice(cfg.S, K_l[h], replace=False)) for h in range(2)]).astype(np.int32)
    k_out = torch.empty((off[-1], cfg.D), dtype=torch.bfloat16, device="cuda")
    v_out = torch.empty_like(k_out)
    pos = torch.empty((off[-1],), dtype=torch.int32, device="cuda")
    K.kvc_gather(inp.k.cuda(), inp.v.cuda(), torch.from_numpy(idx).cuda(), 1, 2, cfg.S, cfg.D, K_l, k_out, v_out, pos)
    K.kvc_check_status()
    for h in range(2):
        sl = slice(off[h], off[h + 1])
        kh, vh, p = O.gather(inp.k[0, h], inp.v[0, h], idx[sl])
        assert torch.equal(k_out[sl].cpu().view(torch.int16), kh.view(torch.int16))
        assert torch.equal(v_out[sl].cpu().view(torch.int16), vh.view(torch.int16))
        assert np.array_equal(pos[sl].cpu().numpy(), p)


def test_run_twice_bitwise_identical(K):
    cfg = small_cfg("gw160_qwen_like")
    inp = make_layer_inputs(cfg)
    K_l, _ = U.kl_vector(cfg, K)
    a = U.run_compress(K, cfg, inp, K_l)
    b = U.run_compress(K, cfg, inp, K_l)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x.view(torch.uint8) if x.dtype != torch.int32 else x,
                           y.view(torch.uint8) if y.dtype != torch.int32 else y)


def test_workspace_does_not_grow_with_S(K):
    """One workspace sized without S serves prompts of 4K and 64K keys."""
    base = dict(H_q=8, H_kv=2, D=128, W=32, pool_k=7, K_l=512, recent=32, hh_frac=0.02)
    ws = K.workspace(1, 8, 2, 128, 32, 4096, 512, 7)
    for S, seed in [(4096, 40), (65536, 41)]:
        cfg = get_config("llama8k", S=S, C=2048, seed=seed, **base)
        inp = make_layer_inputs(cfg)
        K_l, K_l_ref = U.kl_vector(cfg, K)
        k_out, v_out, pos, off = U.run_compress(K, cfg, inp, K_l, ws=ws)
        o = U.oracle_head(cfg, inp, 0, 1)
        U.check_head_outputs(k_out, v_out, pos, off, inp, cfg, 0, 1, K_l_ref[1], o["s"], f"S={S}")


FULL = ["llama8k", "tidekv_main", "mistral128k", "qwen14b"]


def _full_size_heads(cfg, K_l_ref):
    """Heads compared element by element with the oracle at full size: every
    head of the 8K Llama layer (each is small); for Qwen the heads with the
    smallest and the largest budget plus the first and last head; else the
    first and the last head."""
    if cfg.name == "llama8k":
        return [(b, h) for b in range(cfg.B) for h in range(cfg.H_kv)]
    heads = [(0, 0), (cfg.B - 1, cfg.H_kv - 1)]
    if cfg.inverse_stability:
        heads += [(1 % cfg.B, int(np.argmin(K_l_ref))), (2 % cfg.B, int(np.argmax(K_l_ref)))]
    return list(dict.fromkeys(heads))


@pytest.mark.parametrize("name", FULL)
def test_full_size_compress_layer(K, name):
    """Full layer shape, the launch configuration the benchmark times; the
    oracle checks the heads of _full_size_heads, structure every head."""
    cfg = get_config(name)
    layer = 0
    inp = make_layer_inputs(cfg, layer)
    K_l, K_l_ref = U.kl_vector(cfg, K, layer)
    k_out, v_out, pos, off = U.run_compress(K, cfg, inp, K_l, layer=layer)
    U.check_structure_all_heads(pos, off, cfg, K_l_ref)
    for (b, h) in _full_size_heads(cfg, K_l_ref):
        o = U.oracle_head(cfg, inp, b, h)
        U.check_head_outputs(k_out, v_out, pos, off, inp, cfg, b, h, K_l_ref[h], o["s"], f"{name} b={b} h={h}")


@pytest.mark.parametrize("name", FULL)
def test_full_size_scores_sampled_heads(K, name):
    """Element-wise m, Z and pooled scores at full size (the decomposed entry
    points run the same scan kernels as the compress)."""
    cfg = get_config(name)
    inp = make_layer_inputs(cfg)
    K_l, _ = U.kl_vector(cfg, K)
    out = U.run_decomposed(K, cfg, inp, K_l)
    G = cfg.G
    for (b, h) in [(0, 3 % cfg.H_kv), (cfg.B - 1, cfg.H_kv - 1)]:
        o = U.oracle_head(cfg, inp, b, h)
        U.assert_mz_close(out["m"][b, h * G:(h + 1) * G].reshape(-1), out["Z"][b, h * G:(h + 1) * G].reshape(-1),
                          o, f"{name} b={b} h={h}")
        U.assert_scores_close(out["scores"][b, h].numpy(), o["s"], cfg, f"{name} scores b={b} h={h}")
        assert abs(float(out["scores"][b, h].double().sum()) - o["s"].sum()) < 2e-3 * G * cfg.W


@pytest.mark.parametrize("ctas", [1, 2, 3])
def test_all_equal_keys_tie_rule_through_compaction(K, ctas):
    """Every key equal: each window query weighs the keys it sees equally, so
    every interior key gets the same mass and, on the GPU, bit-identical fp32
    scores (one thread per key, the same arithmetic on the same values).  The
    lower index wins ties, so the kept set is exactly the lowest-index
    interior keys, here through the fused path's candidate compaction
    (few scan CTAs, key ranges far longer than K_l_max + b_s)."""
    cfg = get_config("tiny", S=6000, C=6000, H_q=8, H_kv=2, D=128, W=32, pool_k=7, K_l=200, recent=32,
                     b_s=128, hh_frac=0.0, seed=60 + ctas)
    inp = make_layer_inputs(cfg)
    inp.k = inp.k[:, :, :1].expand_as(inp.k).contiguous()      # every key of a head is key 0
    K_l, K_l_ref = U.kl_vector(cfg, K)
    K.kvc_set_option(K.KVC_OPT_SCAN_CTAS, ctas)
    try:
        k_out, v_out, pos, off = U.run_compress(K, cfg, inp, K_l)
    finally:
        K.kvc_set_option(K.KVC_OPT_SCAN_CTAS, 0)
    R = O.mandatory_set(cfg.S, cfg.sink, cfg.recent)
    n_sel = cfg.K_l - len(R)
    want = np.sort(np.concatenate([R, np.arange(cfg.sink, cfg.sink + n_sel)]))
    for h in range(cfg.H_kv):
        got = pos[off[h]:off[h + 1]].numpy()
        assert np.array_equal(got, want), f"ctas={ctas} h={h}: kept {got[cfg.sink:cfg.sink + 8]}..."
        o = U.oracle_head(cfg, inp, 0, h)
        assert np.array_equal(O.select_topk(o["s"], cfg.K_l, cfg.sink, cfg.recent), want)
        U.check_head_outputs(k_out, v_out, pos, off, inp, cfg, 0, h, K_l_ref[h], o["s"], f"all-equal ctas={ctas}")


def test_padded_output_layout_matches_packed(K):
    """A caller's own layout (out_off with room before and between heads):
    select, gather and the whole compress fill the same rows as with the
    packed layout, at the shifted places, and leave the other rows alone."""
    cfg = small_cfg("gw160_qwen_like")            # B = 2, H_kv = 2
    inp = make_layer_inputs(cfg)
    K_l, _ = U.kl_vector(cfg, K)
    K_l = [K_l[0], K_l[1] - 50]
    k_ref, v_ref, p_ref, off = U.run_compress(K, cfg, inp, K_l)
    lay = [5, 5 + K_l[0] + 11, 5 + K_l[0] + 11 + K_l[1] + 3]     # leading gap, gap between, gap at the end
    T = lay[-1]
    q, k, v = U.to_dev(inp)
    ko = torch.full((cfg.B * T, cfg.D), 7.0, dtype=torch.bfloat16, device="cuda")
    vo = torch.full_like(ko, -7.0)
    po = torch.full((cfg.B * T,), -5, dtype=torch.int32, device="cuda")
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, max(K_l), cfg.pool_k)
    K.kvc_compress_layer(cfg.N, 0, cfg.B, cfg.S, cfg.C, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, K_l, cfg.sink,
                         cfg.recent, cfg.pool_k, cfg.b_s, q, k, v, ko, vo, po, ws, out_off=lay)
    K.kvc_check_status()
    ko, vo, po = ko.cpu(), vo.cpu(), po.cpu()
    filled = np.zeros(cfg.B * T, dtype=bool)
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            n = K_l[h]
            a, r = b * T + lay[h], b * off[-1] + off[h]
            filled[a:a + n] = True
            assert torch.equal(po[a:a + n], p_ref[r:r + n]), f"b={b} h={h}: positions"
            assert torch.equal(ko[a:a + n].view(torch.int16), k_ref[r:r + n].view(torch.int16))
            assert torch.equal(vo[a:a + n].view(torch.int16), v_ref[r:r + n].view(torch.int16))
    free = torch.from_numpy(~filled)
    assert torch.all(po[free] == -5) and torch.all(ko[free] == 7.0) and torch.all(vo[free] == -7.0)
    # the decomposed calls with the same layout
    m = torch.empty((cfg.B, cfg.H_q, cfg.W), dtype=torch.float32, device="cuda")
    Z = torch.empty_like(m)
    K.kvc_score_pass1(q, k, cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W, cfg.b_s, m, Z, ws)
    sc = torch.empty((cfg.B, cfg.H_kv, cfg.S), dtype=torch.float32, device="cuda")
    K.kvc_score_pass2_pool(q, k, m, Z, cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W, cfg.b_s, cfg.pool_k, sc, ws)
    idx = torch.full((cfg.B * T,), -9, dtype=torch.int32, device="cuda")
    K.kvc_select_topk(sc, cfg.B, cfg.H_kv, cfg.S, K_l, cfg.sink, cfg.recent, idx, ws, out_off=lay)
    k2 = torch.zeros((cfg.B * T, cfg.D), dtype=torch.bfloat16, device="cuda")
    v2 = torch.zeros_like(k2)
    p2 = torch.full((cfg.B * T,), -5, dtype=torch.int32, device="cuda")
    K.kvc_gather(k, v, idx, cfg.B, cfg.H_kv, cfg.S, cfg.D, K_l, k2, v2, p2, out_off=lay)
    K.kvc_check_status()
    idx, p2 = idx.cpu(), p2.cpu()
    assert torch.all(idx[free] == -9) and torch.all(p2[free] == -5)
    for b in range(cfg.B):
        for h in range(cfg.H_kv):
            a = b * T + lay[h]
            seg = p2[a:a + K_l[h]].numpy().astype(np.int64)
            assert np.array_equal(idx[a:a + K_l[h]].numpy(), seg)
            kh, vh, _ = O.gather(inp.k[b, h], inp.v[b, h], seg)
            assert torch.equal(k2[a:a + K_l[h]].cpu().view(torch.int16), kh.view(torch.int16))
