"""The C-ABI library loads, exports every declared symbol, and its host-only
logic (validation, budgets, layout) behaves as specified.  No GPU work."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O
from synth import get_config, stability_scores

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")


@pytest.fixture(scope="module")
def K():
    from attention_score_kv_gb300 import build
    build.build()
    import attention_score_kv_gb300.kvc as kvc
    return kvc


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kvc_score_pass1", "kvc_score_pass2_pool", "kvc_select_topk", "kvc_gather",
                 "kvc_compress_layer", "kvc_workspace_size"):
        assert must in names


def test_library_exports_every_declared_symbol(K):
    lib = ctypes.CDLL(K.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in kvc.h but not exported"
        assert name in K.EXPORTED, f"{name} has no Python binding"


def test_workspace_size_has_no_S_argument():
    src = open(HEADER).read()
    m = re.search(r"size_t kvc_workspace_size\(([^)]*)\)", src, flags=re.S)
    args = [a.strip().split()[-1] for a in m.group(1).split(",")]
    assert "S" not in args
    assert args == ["B", "H_q", "H_kv", "D", "W", "b_s", "K_l_max", "pool_k"]


def test_version(K):
    assert K.kvc_version() == 300


def test_boundary_takes_the_output_layout():
    """kvc_select_topk, kvc_gather and kvc_compress_layer(_deferred_v) take a
    caller-supplied CSR output layout (const int64_t* out_off), as the
    boundary's call list has them."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for fn in ("kvc_select_topk", "kvc_gather", "kvc_compress_layer", "kvc_compress_layer_deferred_v"):
        m = re.search(fn + r"\(([^)]*)\)", src, flags=re.S)
        assert m and "const int64_t* out_off" in m.group(1), fn


def _call_compress(K, **over):
    a = dict(N=1, layer=0, B=1, S=512, C=512, H_q=4, H_kv=2, D=64, W=16, K_l=[128, 128], sink=4,
             recent=16, pool_k=1, b_s=128, q_win=0x1000, k=0x2000, v=0x3000, k_out=0x4000,
             v_out=0x5000, pos_out=0x6000, ws=0x10000, ws_bytes=1 << 30, stream=0)
    a.update(over)
    return K.kvc_compress_layer(**a)


@pytest.mark.parametrize("over,code", [
    (dict(H_q=5), -1),                 # H_q % H_kv != 0
    (dict(W=600, C=600), -1),          # W > S
    (dict(D=96), -2),                  # unsupported head dim
    (dict(layer=1), -1),               # layer >= N
    (dict(C=8), -1),                   # C < W
    (dict(C=1024), -1),                # C > S
    (dict(pool_k=4), -1),              # even pool
    (dict(pool_k=17), -2),             # pool wider than supported
    (dict(b_s=64), -1),                # block smaller than the scan tile
    (dict(q_win=0), -1),               # null pointer
    (dict(k=0x2004), -1),              # misaligned bf16 tensor
    (dict(H_q=64, H_kv=2, W=16), -2),  # G*W = 512 > 256
    (dict(out_off=[-1, 128, 256]), -1),        # layout starts before row 0
    (dict(out_off=[0, 100, 256]), -1),         # head 0 fills 128 rows, its slot holds 100
    (dict(out_off=[0, 128, 200]), -1),         # the block ends inside head 1's rows
])
def test_compress_layer_rejects_bad_arguments(K, over, code):
    with pytest.raises(K.KvcError) as ei:
        _call_compress(K, **over)
    assert ei.value.code == code


@pytest.mark.parametrize("over,code", [
    (dict(H_q=5), -1),
    (dict(layer=1), -1),
    (dict(C=8), -1),
    (dict(pool_k=4), -1),
    (dict(v=0), -1),
    (dict(k_out=0x4004), -1),
    (dict(D=96), -2),
])
def test_deferred_v_rejects_bad_arguments_before_any_wait(K, over, code):
    """kvc_compress_layer_deferred_v validates like kvc_compress_layer, on the
    host, before it waits on the event or launches anything (the event
    handle here is never touched)."""
    a = dict(N=1, layer=0, B=1, S=512, C=512, H_q=4, H_kv=2, D=64, W=16, K_l=[128, 128], sink=4,
             recent=16, pool_k=1, b_s=128, q_win=0x1000, k=0x2000, v=0x3000, k_out=0x4000,
             v_out=0x5000, pos_out=0x6000, ws=0x10000, v_ready=0x7000, ws_bytes=1 << 30, stream=0)
    a.update(over)
    with pytest.raises(K.KvcError) as ei:
        K.kvc_compress_layer_deferred_v(**a)
    assert ei.value.code == code


def test_budget_below_mandatory_set_is_rejected_before_launch(K):
    # |R_mand| = 4 + 16 = 20 > 19; checked on the host (no device needed to fail)
    with pytest.raises(K.KvcError) as ei:
        K.kvc_select_topk(0x1000, 1, 2, 512, [19, 128], 4, 16, 0x2000, 0x10000, 1 << 20, stream=0)
    assert ei.value.code == -1
    with pytest.raises(K.KvcError) as ei:    # overlapping head slots
        K.kvc_select_topk(0x1000, 1, 2, 512, [128, 128], 4, 16, 0x2000, 0x10000, 1 << 20, stream=0,
                          out_off=[0, 64, 300])
    assert ei.value.code == -1
    with pytest.raises(K.KvcError) as ei:    # a gather layout that cannot hold head 1's rows
        K.kvc_gather(0x1000, 0x2000, 0x3000, 1, 2, 512, 64, [128, 128], 0x4000, 0x5000, 0x6000, stream=0,
                     out_off=[0, 128, 255])
    assert ei.value.code in (-1, -4)


def test_select_null_scores(K):
    with pytest.raises(K.KvcError) as ei:
        K.kvc_select_topk(0, 1, 2, 512, [128, 128], 4, 16, 0x2000, 0x10000, 1 << 20, stream=0)
    assert ei.value.code == -1


def test_budgets_match_oracle_bit_exact(K):
    cfg = get_config("qwen14b")
    total = round(cfg.budget_frac * cfg.S * cfg.H_kv)
    rsz = cfg.sink + cfg.recent
    for layer in range(48):
        s = stability_scores(cfg, layer).numpy()
        got = K.kvc_budget_inverse_stability(s, total, rsz, cfg.S)
        exp = O.budgets_inverse_stability(s, total, rsz, cfg.S)
        assert got == exp.tolist()
        assert sum(got) == total
    # clamp and tie cases
    assert K.kvc_budget_inverse_stability([1.0, 1.0, 0.01], 300, 50, 200) == \
        O.budgets_inverse_stability([1.0, 1.0, 0.01], 300, 50, 200).tolist()
    assert K.kvc_budget_inverse_stability([1.0] * 3, 10, 0, 100) == [4, 3, 3]
    assert K.kvc_budget_inverse_stability([1.0, 2.0, 4.0], 10, 0, 100) == [6, 3, 1]   # worked by hand
    # The host function rounds in fp64 and the oracle in exact rationals; they
    # can only disagree where two remainders lie within fp64 rounding of each
    # other, which none of these draws comes near.
    rng = np.random.default_rng(0)
    for _ in range(200):
        H = int(rng.integers(1, 17))
        s = rng.uniform(0.01, 1.0, H)
        total = int(rng.integers(0, 100000))
        assert K.kvc_budget_inverse_stability(s, total, 0, 1 << 30) == \
            O.budgets_inverse_stability(s, total, 0, 1 << 30).tolist()


def test_retained_layout_matches_oracle(K):
    for S, kl in [(100, [10, 200, 5]), (512, [128, 128]), (32768, [4096] * 8)]:
        assert K.kvc_retained_layout(len(kl), S, kl) == O.retained_layout(S, kl).tolist()


def test_main_config_retained_cache_is_512_mib(K):
    cfg = get_config("tidekv_main")
    off = K.kvc_retained_layout(cfg.H_kv, cfg.S, [cfg.K_l] * cfg.H_kv)
    per_layer = off[-1] * cfg.B * cfg.D * 2 * 2      # K and V, bf16
    assert per_layer * cfg.N == 512 * 2**20


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """Importing the binding with no libkvc.so raises instead of falling back."""
    import importlib.util
    src = os.path.join(ROOT, "attention_score_kv_gb300", "kvc.py")
    dst = tmp_path / "kvc.py"
    dst.write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("kvc_copy", dst)
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_product_does_not_import_oracle():
    pkg = os.path.join(ROOT, "attention_score_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.sub(r"(#|//).*", "", txt), f"{f} mentions the oracle"


@pytest.mark.parametrize("N,budget,k_min", [(32, 4096, 1024), (48, 256, 36), (7, 1000, 1000), (1, 512, 100),
                                            (5, 33, 7)])
def test_pyramid_budgets_match_oracle(K, N, budget, k_min):
    from oracle import layer_major as LM
    assert K.kvc_budget_pyramid(N, budget, k_min) == LM.budgets_pyramid(N, budget, k_min)
    with pytest.raises(K.KvcError):
        K.kvc_budget_pyramid(4, 10, 11)


def test_cache_layout_matches_oracle(K):
    from oracle import layer_major as LM
    K_l = [[100, 300, 9000], [64, 64, 64], [0, 1, 2]]
    assert K.kvc_cache_layout(3, 2, 3, 8192, K_l) == LM.cache_layout(3, 2, 8192, K_l).tolist()


def _ranges_cases():
    rng = np.random.default_rng(7)
    cases = [(8, 131072, 152), (8, 65536, 152), (32, 32768, 152), (8, 8192, 152), (2, 700, 6), (2, 700, 9),
             (4, 700, 3), (4, 700, 5), (1, 512, 152), (1, 1, 1), (3, 1000, 1), (16, 777, 152)]
    for _ in range(200):
        cases.append((int(rng.integers(1, 40)), int(rng.integers(1, 300000)), int(rng.integers(1, 200))))
    return cases


def test_scan_ranges_cover_the_keys_and_snap_to_heads(K):
    """The CTA key ranges of the scans: ordered, non-empty, covering [0, BH*S)
    exactly; a cut within min(L/4, 512) keys of a head boundary sits on it,
    every other cut stays at c * L; a range is at most 2 * snap keys longer
    than L and at least L / 2 long."""
    for BH, S, P in _ranges_cases():
        total = BH * S
        st = K.kvc_scan_ranges(BH, S, P)
        n = len(st) - 1
        assert 1 <= n <= P
        L = -(-total // min(P, total))
        assert n == -(-total // L)
        snap = min(L // 4, 512)
        assert st[0] == 0 and st[-1] == total
        for c in range(n):
            assert st[c + 1] > st[c], (BH, S, P, c)
            assert L // 2 <= st[c + 1] - st[c] <= L + 2 * snap or c == n - 1, (BH, S, P, c)
        for c in range(1, n):
            f, r = c * L, (c * L) % S
            if r != 0 and (r <= snap or S - r <= snap):
                assert st[c] % S == 0 and abs(st[c] - f) <= snap, (BH, S, P, c, st[c], f)
            else:
                assert st[c] == f, (BH, S, P, c, st[c], f)


def test_scan_ranges_mistral_layer_has_no_two_head_range(K):
    """Mistral-7B at S = 131072 on 152 CTAs: every range lies inside one KV
    head (the unsnapped cut gave 7 CTAs a 9-63-key sliver of the next head)."""
    S = 131072
    st = K.kvc_scan_ranges(8, S, 152)
    assert len(st) == 153
    for a, b in zip(st[:-1], st[1:]):
        assert a // S == (b - 1) // S


def test_scan_ranges_rejects_bad_sizes(K):
    for args in ((0, 10, 1), (1, 0, 1), (1, 10, 0)):
        with pytest.raises(K.KvcError):
            K.kvc_scan_ranges(*args)


def test_budget_helpers_reject_overflowing_inputs(K):
    # a first-layer budget 2*budget - k_min past int32 cannot be returned
    with pytest.raises(K.KvcError) as ei:
        K.kvc_budget_pyramid(4, 2**31 - 2, 0)
    assert ei.value.code == K.KVC_ERR_INVALID_ARG
    assert K.kvc_budget_pyramid(2, 2**30, 1) == [2**31 - 1, 1]        # the largest that fits
    # a positive but subnormal stability score makes 1/s overflow fp64
    for s in ([1.0, 1e-310], [1e-308, 1e-308], [1e-300, 1.0]):
        with pytest.raises(K.KvcError) as ei:
            K.kvc_budget_inverse_stability(s, 10**12 if s[0] == 1e-300 else 100, 0, 1 << 30)
        assert ei.value.code == K.KVC_ERR_INVALID_ARG
    # tiny but representable scores still work and match the oracle
    s = [1e-200, 1.0, 2.0]
    assert K.kvc_budget_inverse_stability(s, 1000, 0, 1 << 30) == \
        O.budgets_inverse_stability(s, 1000, 0, 1 << 30).tolist()


def test_workspace_rejects_a_key_block_that_would_overflow_the_candidate_capacity(K):
    # checked before the device is asked for its SM count, so no GPU is needed
    with pytest.raises(K.KvcError) as ei:
        K.kvc_workspace_size(1, 4, 2, 64, 16, 2**29 + 1, 100, 1)
    assert "b_s" in str(ei.value)
    with pytest.raises(K.KvcError) as ei:
        K.kvc_workspace_size(1, 4, 2, 64, 16, 127, 100, 1)
    assert "b_s" in str(ei.value)
