"""The allocation-free pass 1 (kvc_score_pass1_noalloc) against the
workspace version, through the C ABI.

kvc_score_pass1_noalloc serves callers that may not allocate device memory
(a host framework that owns all device memory in its own pool, or plugin and
real-time paths that may not call the CUDA allocator); it keeps its scratch
in a fixed array inside the library.  This file is collected last so that a
run stopping at the first failure has already run every other test.
"""

import pytest
import torch

from synth import get_config, make_layer_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_score_kv_gb300 import build
    build.build()
    import attention_score_kv_gb300.kvc as kvc
    return kvc


def _pass1_with_workspace(K, cfg, q, k):
    ws = K.workspace(cfg.B, cfg.H_q, cfg.H_kv, cfg.D, cfg.W, cfg.b_s, 0, 1)
    m = torch.empty((cfg.B, cfg.H_q, cfg.W), dtype=torch.float32, device="cuda")
    Z = torch.empty_like(m)
    K.kvc_score_pass1(q, k, cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W, cfg.b_s, m, Z, ws)
    return m, Z


def _pass1_noalloc(K, cfg, q, k):
    m = torch.full((cfg.B, cfg.H_q, cfg.W), float("nan"), dtype=torch.float32, device="cuda")
    Z = torch.full_like(m, float("nan"))
    K.kvc_score_pass1_noalloc(q, k, cfg.B, cfg.H_q, cfg.H_kv, cfg.S, cfg.D, cfg.W, cfg.b_s, m, Z)
    return m, Z


def _close(a, b):
    a, b = a.double(), b.double()
    return bool(torch.all((a - b).abs() <= TOL * torch.clamp(b.abs(), min=1.0)))


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("llama8k", {}),
    ("tiny", dict(B=2, S=3000, C=3000, H_q=10, H_kv=2, D=128, W=32, seed=7)),
])
def test_noalloc_pass1_matches_workspace_pass1_twice(K, name, over):
    """These shapes fit the default key-range plan, so both entry points run
    the same kernels over the same ranges: m and Z must be bit-identical."""
    cfg = get_config(name, **over)
    inp = make_layer_inputs(cfg)
    q, k = inp.q_win.cuda(), inp.k.cuda()
    m_ref, Z_ref = _pass1_with_workspace(K, cfg, q, k)
    for call in range(2):                      # two calls in a row share the array
        m, Z = _pass1_noalloc(K, cfg, q, k)
        K.kvc_check_status()
        assert torch.equal(m, m_ref), f"call {call}: m differs"
        assert torch.equal(Z, Z_ref), f"call {call}: Z differs"


def test_noalloc_pass1_one_range_per_head_plan(K):
    """500 heads of 256 window rows: the default plan's partials (152 ranges,
    each touching up to 4 heads: 1.2 MiB) do not fit the fixed array, so the
    call falls back to one key range per head (1,024,000 bytes).  Different
    ranges round differently, so the results agree within the scorer's
    tolerance, on two calls in a row."""
    cfg = get_config("tiny", B=125, H_q=32, H_kv=4, D=64, S=768, C=768, W=32, seed=11)
    inp = make_layer_inputs(cfg)
    q, k = inp.q_win.cuda(), inp.k.cuda()
    m_ref, Z_ref = _pass1_with_workspace(K, cfg, q, k)
    for call in range(2):
        m, Z = _pass1_noalloc(K, cfg, q, k)
        K.kvc_check_status()
        assert _close(m, m_ref), f"call {call}: m differs"
        assert _close(Z, Z_ref), f"call {call}: Z differs"


def test_noalloc_pass1_alternating_shapes(K):
    """A smaller call after a larger one must not see the larger call's leftovers."""
    big = get_config("llama8k")
    small = get_config("tiny")
    ib, is_ = make_layer_inputs(big), make_layer_inputs(small)
    qb, kb = ib.q_win.cuda(), ib.k.cuda()
    qs, ks = is_.q_win.cuda(), is_.k.cuda()
    ref_b = _pass1_with_workspace(K, big, qb, kb)
    ref_s = _pass1_with_workspace(K, small, qs, ks)
    for cfg, q, k, ref in [(big, qb, kb, ref_b), (small, qs, ks, ref_s), (big, qb, kb, ref_b)]:
        m, Z = _pass1_noalloc(K, cfg, q, k)
        assert _close(m, ref[0]) and _close(Z, ref[1])
    K.kvc_check_status()


def test_noalloc_rejects_shapes_beyond_the_fixed_array(K):
    # B * H_kv * roundup16(G*W) * 8 bytes = 1024 * 256 * 8 = 2 MiB > 1 MiB.
    # The tensors are real and of the stated shapes, so that even a broken
    # size check would only run a valid pass 1 (and fail the test), never
    # read or write outside an allocation.
    B, H_q, H_kv, S, D, W = 1024, 1, 1, 512, 64, 256
    q = torch.zeros((B, H_q, W, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, H_kv, S, D), dtype=torch.bfloat16, device="cuda")
    m = torch.zeros((B, H_q, W), dtype=torch.float32, device="cuda")
    Z = torch.zeros_like(m)
    with pytest.raises(K.KvcError) as ei:
        K.kvc_score_pass1_noalloc(q, k, B, H_q, H_kv, S, D, W, 128, m, Z)
    assert ei.value.code == K.KVC_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)
    K.kvc_check_status()
