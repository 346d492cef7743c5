"""Pins of the low-rank gate predictor's oracle (oracle/predictor.py), CPU."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from oracle import predictor as P
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import ffn_from_layer, mat_from_act, mat_from_weight


def _layer(F=96, d=64, seed=5):
    return W.make_ffn_layer(2, seed=seed, d_model=d, d_ff=F)


def test_infinite_margin_is_the_exact_decode():
    layer = _layer()
    ffn, x = ffn_from_layer(layer), mat_from_act(W.make_tokens(2, 6, seed=1, d_model=64))
    A, B = P.lowrank_factors(mat_from_weight(layer, "gate").to_f64(), 8)
    r = P.decode_predicted(ffn, x, A, B, np.inf)
    ref = O.decode(ffn, x, O.EXACT)
    assert np.array_equal(r["out"], ref["out"])              # same set, same arithmetic
    for t in range(6):
        assert r["candidates"][t].size == 96
        assert np.array_equal(r["active"][t], ref["active_idx"][t, : ref["n_active"][t]])
    assert np.all(r["recall"] == 1.0)


def test_no_candidate_gives_zero_output():
    layer = _layer()
    ffn, x = ffn_from_layer(layer), mat_from_act(W.make_tokens(2, 4, seed=2, d_model=64))
    A, B = P.lowrank_factors(mat_from_weight(layer, "gate").to_f64(), 4)
    r = P.decode_predicted(ffn, x, A, B, -np.inf)
    assert not r["out"].any() and all(c.size == 0 for c in r["candidates"])


def test_full_rank_factors_reproduce_the_gate():
    layer = _layer(F=80, d=48)
    Wg = mat_from_weight(layer, "gate").to_f64()
    A, B = P.lowrank_factors(Wg, 48)
    assert np.abs(A @ B - Wg).max() < 1e-12
    x = W.make_tokens(2, 5, seed=3, d_model=48)
    ffn, xm = ffn_from_layer(layer), mat_from_act(x)
    ref = O.decode(ffn, xm, O.EXACT, details=True)
    p = P.predict(A, B, layer["b_gate"].numpy(), xm.to_f64())
    assert np.abs(p - ref["g"]).max() < 1e-10
    r = P.decode_predicted(ffn, xm, A, B, 1e-9)
    assert np.all(r["recall"] == 1.0)


def test_exact_low_rank_gate_is_predicted_without_misses():
    # a gate of exact rank 6: the rank-6 predictor finds every active neuron and,
    # at a vanishing margin, nothing else
    F, d, r = 96, 64, 6
    layer = _layer(F=F, d=d)
    g = torch.Generator().manual_seed(9)
    Wg = (torch.randn(F, r, generator=g) @ torch.randn(r, d, generator=g)) / np.sqrt(d * r)
    layer["w_gate"] = Wg.to(torch.bfloat16)
    Wq = mat_from_weight(layer, "gate").to_f64()            # the bf16 matrix is no longer exactly rank 6
    A, B = P.lowrank_factors(Wq, F)                           # so compare against full rank ...
    A6, B6 = P.lowrank_factors(Wg.double().numpy(), r)        # ... and the rank-6 factors of the exact matrix
    ffn, x = ffn_from_layer(layer), mat_from_act(W.make_tokens(2, 8, seed=4, d_model=d))
    full = P.decode_predicted(ffn, x, A, B, 1e-9)
    assert np.all(full["recall"] == 1.0)
    six = P.decode_predicted(ffn, x, A6, B6, 0.05)            # margin covers the bf16 rounding of the gate
    assert np.all(six["recall"] == 1.0)


def test_candidates_grow_with_the_margin():
    layer = _layer(seed=11)
    ffn, x = ffn_from_layer(layer), mat_from_act(W.make_tokens(2, 3, seed=5, d_model=64))
    A, B = P.lowrank_factors(mat_from_weight(layer, "gate").to_f64(), 4)
    prev = None
    for alpha in (0.0, 0.05, 0.2, 1.0, np.inf):
        r = P.decode_predicted(ffn, x, A, B, alpha)
        if prev is not None:
            for t in range(3):
                assert set(prev["candidates"][t]) <= set(r["candidates"][t])
                assert r["recall"][t] >= prev["recall"][t]
                assert r["bytes"][t] >= prev["bytes"][t]
        prev = r


def test_byte_count():
    layer = _layer()
    ffn, x = ffn_from_layer(layer), mat_from_act(W.make_tokens(2, 2, seed=6, d_model=64))
    A, B = P.lowrank_factors(mat_from_weight(layer, "gate").to_f64(), 4)
    r = P.decode_predicted(ffn, x, A, B, np.inf)
    for t in range(2):
        n = r["active"][t].size
        assert r["bytes"][t] == pytest.approx(2.0 * (96 * 64 + 2 * n * 64) + 4.0 * 4 * (96 + 64))
