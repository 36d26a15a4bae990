"""GPU parity of HeteroCache's overlap coefficient, head similarity and
device budgets, through the C ABI.  The overlap is an exact integer ratio
divided once in float32 and the budgets repeat the host's float64 steps, so
everything must match bit for bit."""

import numpy as np
import pytest
import torch

from oracle import heterocache as Hc
from oracle import kvc_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import attention_score_kv_gb300.kvc as K
    return K


def _csr(sets):
    off = np.concatenate([[0], np.cumsum([len(s) for s in sets])]).astype(np.int64)
    flat = np.concatenate([np.asarray(s, dtype=np.int32) for s in sets]) if off[-1] else np.zeros(1, np.int32)
    return torch.from_numpy(flat).cuda(), torch.from_numpy(off).cuda()


def test_overlap_pairs_bit_exact(K):
    rng = np.random.default_rng(0)
    A, B = [], []
    for i in range(300):
        n = int(rng.integers(0, 5000)) if i % 17 else 0             # some empty sets
        m = int(rng.integers(1, 5000))
        A.append(np.sort(rng.choice(131072, n, replace=False)))
        B.append(np.sort(np.concatenate([A[-1][: n // 3], rng.choice(131072, m, replace=False)])))
        B[-1] = np.unique(B[-1])
    A[5] = B[5].copy()                                               # identical
    a, a_off = _csr(A)
    b, b_off = _csr(B)
    out = torch.empty(len(A), dtype=torch.float32, device="cuda")
    K.kvc_overlap_coefficient(a, a_off, b, b_off, len(A), out)
    K.kvc_check_status()
    got = out.cpu().numpy()
    ref = np.array([Hc.overlap_coefficient(x, y) for x, y in zip(A, B)], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert got[5] == 1.0


def test_similarity_of_selected_sets_bit_exact(K):
    # the sets kvc_select_topk writes, for 2 groups of 8 heads
    rng = np.random.default_rng(1)
    B, H, S = 2, 8, 20000
    s = rng.standard_normal((B, H, S)).astype(np.float32)
    s[:, 3] = s[:, 2] + 0.01 * rng.standard_normal((B, S)).astype(np.float32)   # two similar heads
    K_l = [1000 + 100 * h for h in range(H)]
    idx = torch.empty((B, sum(K_l)), dtype=torch.int32, device="cuda")
    ws = K.workspace(B, H, H, 64, 1, 128, max(K_l), 1, device="cuda")
    K.kvc_select_topk(torch.from_numpy(s).cuda(), B, H, S, K_l, 4, 16, idx, ws)
    offs = np.concatenate([[0], np.cumsum(K_l)])
    off = np.stack([offs + g * offs[-1] for g in range(B)]).astype(np.int64)
    sim = torch.empty(B * H, dtype=torch.float32, device="cuda")
    K.kvc_head_similarity(idx.reshape(-1), torch.from_numpy(off).cuda(), B, H, sim)
    K.kvc_check_status()
    got = sim.cpu().numpy()
    flat = idx.cpu().numpy().reshape(-1)
    for g in range(B):
        sets = [flat[off[g, i]:off[g, i + 1]] for i in range(H)]
        ref = Hc.head_similarity(sets)
        assert np.array_equal(got[g * H:(g + 1) * H].view(np.uint32), ref.view(np.uint32)), g
        assert got[g * H + 2] > 0.5 and got[g * H + 3] > 0.5


def test_device_budgets_equal_host_and_oracle(K):
    rng = np.random.default_rng(2)
    n_layers, H = 48, 8
    s = rng.uniform(0.2, 1.0, (n_layers, H))
    s[7] = 0.5                                                       # equal scores: remainders tie
    total, lo, hi = 78643, 68, 32768
    out = torch.empty((n_layers, H), dtype=torch.int32, device="cuda")
    K.kvc_budget_inverse_stability_device(n_layers, H, torch.from_numpy(s).cuda(), total, lo, hi, out)
    K.kvc_check_status()
    got = out.cpu().numpy()
    for l in range(n_layers):
        assert got[l].tolist() == K.kvc_budget_inverse_stability(s[l], total, lo, hi), l
        assert got[l].tolist() == O.budgets_inverse_stability(s[l], total, lo, hi).tolist(), l


def _drifting_sets(rng, T, H, S, k, drift):
    """Seeded synthetic decoding-step top-k sets: each head starts from its
    prefill set and replaces a head-specific share of it at every step."""
    pre = [np.sort(rng.choice(S, k, replace=False)) for _ in range(H)]
    dec = []
    for t in range(T):
        row = []
        for h in range(H):
            keep = rng.random(k) >= drift[h]
            new = rng.choice(S, int((~keep).sum()), replace=False)
            row.append(np.unique(np.concatenate([pre[h][keep], new])))
        dec.append(row)
    return pre, dec


@pytest.mark.parametrize("T", [1, 100, 101])
def test_phase1_medians_over_steps_bit_exact(K, T):
    """HeteroCache Phase 1: stability = median over T steps of the overlap of
    each head's step set with its prefill set; similarity = median over the
    steps of the per-step maximum overlap with another head."""
    rng = np.random.default_rng(T)
    H, S, k = 8, 32768, 512
    drift = np.linspace(0.02, 0.9, H)
    pre, dec = _drifting_sets(rng, T, H, S, k, drift)
    flat_dec = [dec[t][h] for t in range(T) for h in range(H)]
    d_idx, d_off = _csr(flat_dec)
    p_idx, p_off = _csr(pre)
    per = torch.empty((T, H), dtype=torch.float32, device="cuda")
    stab = torch.empty(H, dtype=torch.float32, device="cuda")
    K.kvc_head_stability_over_steps(d_idx, d_off, p_idx, p_off, T, H, per, stab)
    # similarity: each step a group of H sets with its own CSR offsets
    offs = [np.concatenate([[0], np.cumsum([len(x) for x in dec[t]])]) for t in range(T)]
    base = np.cumsum([0] + [o[-1] for o in offs[:-1]])
    off2 = torch.from_numpy(np.stack([o + b for o, b in zip(offs, base)]).astype(np.int64)).cuda()
    per2 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    sim = torch.empty(H, dtype=torch.float32, device="cuda")
    K.kvc_head_similarity_over_steps(d_idx, off2, T, H, per2, sim)
    K.kvc_check_status()
    ref_per, ref_stab = Hc.stability_over_steps(dec, pre)
    ref_per2, ref_sim = Hc.similarity_over_steps(dec)
    assert np.array_equal(per.cpu().numpy().view(np.uint32), ref_per.view(np.uint32))
    assert np.array_equal(stab.cpu().numpy().view(np.uint32), ref_stab.view(np.uint32))
    assert np.array_equal(per2.cpu().numpy().view(np.uint32), ref_per2.view(np.uint32))
    assert np.array_equal(sim.cpu().numpy().view(np.uint32), ref_sim.view(np.uint32))
    if T > 1:   # slow drift gives the higher stability
        assert np.all(np.diff(ref_stab) <= 0)


def test_median_over_steps_ties_and_signs(K):
    x = np.array([[0.25, -0.0, 1.0], [0.25, 0.0, 2.0], [0.5, -0.0, 3.0], [0.75, 5.0, 4.0]], dtype=np.float32)
    for T in (1, 2, 3, 4):
        med = torch.empty(3, dtype=torch.float32, device="cuda")
        K.kvc_median_over_steps(torch.from_numpy(x[:T].copy()).cuda(), T, 3, med)
        K.kvc_check_status()
        ref = Hc.median_over_steps(x[:T])
        assert np.array_equal(med.cpu().numpy().view(np.uint32), ref.view(np.uint32)), T
