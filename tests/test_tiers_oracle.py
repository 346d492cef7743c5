"""Pins of the tier-table oracle (oracle/tiers.py): a core set per layer and tier,
completed per token by the largest remaining scores.  CPU."""
from __future__ import annotations

import itertools

import numpy as np

import oracle as O
from oracle import tiers as T
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import ffn_from_layer, mat_from_act


def test_empty_core_is_the_keep_ratio_selection():
    layer = W.make_ffn_layer(3, seed=21, d_model=64, d_ff=96)
    ffn = ffn_from_layer(layer)
    x = mat_from_act(W.make_tokens(3, 5, seed=2, d_model=64))
    for ratio in (0.5, 0.25, 0.125):
        ref = O.decode(ffn, x, O.KEEP_RATIO, O.SCORE_GATE_UP, ratio, details=True)
        k = O.keep_count(96, ratio)
        for t in range(5):
            want = ref["active_idx"][t, : ref["n_active"][t]]
            got = T.select_with_core(ref["score"][t], k, np.zeros(0, np.int32))
            assert np.array_equal(got, want)


def test_full_core_is_returned_as_is():
    rng = np.random.default_rng(0)
    s = rng.random(40)
    core = np.array([1, 5, 9, 33], np.int32)
    assert np.array_equal(T.select_with_core(s, 4, core), core)


def test_brute_force_on_small_layers():
    # the selection maximises the kept score among all size-k sets that contain
    # the core (distinct scores: unique maximiser)
    rng = np.random.default_rng(1)
    for F in (6, 9, 11):
        for trial in range(6):
            s = rng.permutation(F).astype(np.float64) + rng.random(F) * 0.1
            k = int(rng.integers(1, F))
            c = int(rng.integers(0, k + 1))
            core = np.sort(rng.choice(F, c, replace=False)).astype(np.int32)
            best, best_sum = None, -1.0
            rest = [j for j in range(F) if j not in set(core.tolist())]
            for extra in itertools.combinations(rest, k - c):
                tot = s[list(extra)].sum() + s[core].sum()
                if tot > best_sum:
                    best, best_sum = np.sort(np.concatenate([core, np.array(extra, np.int32)])), tot
            assert np.array_equal(T.select_with_core(s, k, core), best)


def test_ties_go_to_the_lower_index():
    s = np.ones(10)
    assert T.select_with_core(s, 3, np.array([7], np.int32)).tolist() == [0, 1, 7]
    assert T.topk_lower_index(s, 4).tolist() == [0, 1, 2, 3]


def test_core_set_counts_frequencies():
    # columns 2 and 5 are in every calibration token's top-2; column 8 in half
    F, N = 10, 8
    S = np.zeros((N, F))
    S[:, 2] = 5.0
    S[:, 5] = 4.0
    S[::2, 8] = 6.0           # tokens 0, 2, 4, 6: top-2 = {8, 2}; tokens 1, 3, 5, 7: {2, 5}
    assert T.core_set(S, 2, 1).tolist() == [2]        # kept 8 times
    got = T.core_set(S, 2, 2)
    # frequencies: 2 -> 8, 5 -> 4, 8 -> 4: the tie between 5 and 8 goes to 5
    assert got.tolist() == [2, 5]
    assert T.core_set(S, 2, 3).tolist() == [2, 5, 8]
    assert T.core_set(S, 2, 0).size == 0


def test_core_then_supplement_keeps_k_per_token():
    rng = np.random.default_rng(3)
    F, k = 64, 16
    calib = rng.random((20, F)) * np.linspace(2.0, 1.0, F)   # earlier columns score higher on average
    core = T.core_set(calib, k, 8)
    for t in range(10):
        sel = T.select_with_core(rng.random(F), k, core)
        assert sel.size == k and np.all(np.diff(sel) > 0) and set(core.tolist()) <= set(sel.tolist())
