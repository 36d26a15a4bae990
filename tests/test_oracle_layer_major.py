"""Pins of the layer-major prefill oracle (CPU only): chunks reassemble the
prompt, and the cross-layer cache at TideKV's main setting is the 512 MiB the
pages report."""

import json
import os

import numpy as np
import pytest

from oracle import layer_major as LM


@pytest.mark.parametrize("S,C", [(700, 128), (512, 128), (5, 8), (1, 1)])
def test_chunks_reassemble_the_prompt(S, C):
    rng = np.random.default_rng(S)
    full = rng.standard_normal((2, 3, S, 4)).astype(np.float32)
    bounds = LM.chunk_bounds(S, C)
    assert bounds[0][0] == 0 and bounds[-1][1] == S
    assert all(b - a == C for a, b in bounds[:-1]) and 0 < bounds[-1][1] - bounds[-1][0] <= C
    chunks = [full[:, :, a:b] for a, b in bounds]
    assert np.array_equal(LM.assemble_chunks(chunks, S), full)


def test_main_setting_cache_is_512_mib(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "retained_cache_512mib.json")))
    N, H, K_l, D, B = g["N"], g["H_kv"], g["K_l"], g["D"], g["B"]
    off = LM.cache_layout(N, B, 65536, [[K_l] * H] * N)
    assert off[-1] * D * g["elem_bytes"] * 2 == g["bytes"]     # K^ and V^ rows of all layers


def test_layout_of_unequal_layers():
    K_l = [[10, 20, 600], [1, 2, 3]]           # the 600 is clamped to S = 500
    off = LM.cache_layout(2, 3, 500, K_l)
    assert off.tolist() == [0, 3 * (10 + 20 + 500), 3 * 530 + 3 * 6]


@pytest.mark.parametrize("N,budget,k_min", [(32, 4096, 1024), (48, 256, 36), (7, 1000, 1000), (1, 512, 100),
                                            (2, 10, 3), (40, 1024, 0)])
def test_pyramid_budgets_sum_ends_and_shape(N, budget, k_min):
    b = LM.budgets_pyramid(N, budget, k_min)
    assert len(b) == N and sum(b) == N * budget                    # the average budget holds exactly
    assert all(x >= y for x, y in zip(b, b[1:]))                    # shrinks with depth
    if N > 1:
        assert abs(b[0] - (2 * budget - k_min)) <= 1 and abs(b[-1] - k_min) <= 1
    if k_min == budget:
        assert b == [budget] * N                                    # no ramp: flat


@pytest.mark.parametrize("N,budget,k_min,expected", [
    # worked by hand from the reading (a linear ramp from 2*budget - k_min down
    # to k_min, largest-remainder rounding, equal remainders to the lower layer):
    (2, 10, 3, [17, 3]),            # ends only
    (4, 10, 1, [19, 13, 7, 1]),     # integer steps of 6
    (4, 5, 0, [10, 7, 3, 0]),       # 10, 6.67, 3.33, 0: the one spare key goes to the largest remainder
    (5, 4, 1, [7, 6, 4, 2, 1]),     # 7, 5.5, 4, 2.5, 1: remainders tie at layers 1 and 3, the lower one wins
])
def test_pyramid_budgets_hand_cases(N, budget, k_min, expected):
    assert LM.budgets_pyramid(N, budget, k_min) == expected


@pytest.mark.parametrize("N,budget,k_min", [(32, 4096, 1024), (48, 256, 36), (9, 100, 7), (40, 1024, 0)])
def test_pyramid_budgets_stay_within_one_key_of_the_linear_ramp(N, budget, k_min):
    from fractions import Fraction
    b = LM.budgets_pyramid(N, budget, k_min)
    k_max = 2 * budget - k_min
    for l, x in enumerate(b):
        exact = Fraction(k_max) - Fraction((k_max - k_min) * l, N - 1)
        assert abs(Fraction(x) - exact) < 1
