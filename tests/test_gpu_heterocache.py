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
