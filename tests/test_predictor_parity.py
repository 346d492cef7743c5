"""GPU parity of sffn_decode_predicted (the low-rank gate predictor) against the
fp64 oracle (oracle/predictor.py) on the same fp32 factors.

The active set is bit-exact except for neurons within a rounding band of one of
the two decisions: the candidate test p_j >= -alpha (band: 1e-5 of the sum of
the magnitudes that form p_j, which bounds the fp32 error of B x and of A y),
and the exact rule act(g_j) != 0 (the decode's tie band).  At most two such
neurons per token are forgiven.  The output is compared with the oracle's
output on the GPU's own set at the decode's tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from oracle import predictor as P
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import ffn_from_layer, mat_from_act, mat_from_weight
from tests.parity import TIE_REL, TOL, check_outputs, layer_to

pytestmark = pytest.mark.gpu

P_BAND = 1e-5


@pytest.fixture(scope="module")
def S():
    from activation_sparse_ffn_gemv_gb300 import build as B
    B.build()
    from activation_sparse_ffn_gemv_gb300 import sffn
    sffn.lib()
    return sffn


def _svd_factors(layer, r):
    A, B = P.lowrank_factors(mat_from_weight(layer, "gate").to_f64(), r)
    return A.astype(np.float32), B.astype(np.float32)


def _random_factors(F, d, r, seed, x=None, sd=0.5):
    """Gaussian factors; with x given, A is scaled so that A (B x) has standard
    deviation `sd` (the spread of the gate bias around its mean)."""
    g = np.random.default_rng(seed)
    A = g.standard_normal((F, r)) / np.sqrt(r)
    B = (g.standard_normal((r, d)) / np.sqrt(d)).astype(np.float32)
    if x is not None:
        p = A @ (B.astype(np.float64) @ mat_from_act(x).to_f64()[0])
        A = A * (sd / p.std())
    return A.astype(np.float32), B


def _alpha_for(layer, x_cpu, A, B, frac):
    """alpha that makes about `frac` of the neurons candidates, with -alpha
    midway across the widest gap between neighbouring predicted values near
    that quantile (so no value lies at the cut)."""
    bias = None if layer.get("b_gate") is None else layer["b_gate"].double().numpy()
    p = P.predict(A.astype(np.float64), B.astype(np.float64), bias, mat_from_act(x_cpu).to_f64())[0]
    s = np.sort(p)[::-1]
    k0 = max(1, min(s.size - 1, int(frac * s.size)))
    ks = range(k0, min(s.size, k0 + 64))
    k = max(ks, key=lambda kk: s[kk - 1] - s[kk])
    cut = 0.5 * (s[k - 1] + s[k])
    assert cut < 0.0, "the quantile lies above zero: alpha >= 0 cannot express it"
    return float(-cut)


def run_and_check(S, layer_cpu, x_cpu, A, B, alpha, max_exempt=2):
    dev = "cuda"
    w = S.Weights(layer_to(layer_cpu, dev))
    x = x_cpu.to(dev)
    fa = None if A is None else torch.from_numpy(A).to(dev)
    fb = None if B is None else torch.from_numpy(B).to(dev)
    out, idx, n = S.decode_predicted(x, w, fa, fb, alpha)
    torch.cuda.synchronize()
    nn = int(n.item())
    gs = idx[0, :nn].cpu().numpy()
    F = layer_cpu["d_ff"]
    assert gs.size == 0 or (np.all(np.diff(gs) > 0) and gs[0] >= 0 and gs[-1] < F)
    ffn, xm = ffn_from_layer(layer_cpu), mat_from_act(x_cpu)
    r = F if A is None else A.shape[1]
    A64 = np.zeros((F, r)) if A is None else A.astype(np.float64)
    B64 = np.zeros((r, layer_cpu["d_model"])) if B is None else B.astype(np.float64)
    ref = P.decode_predicted(ffn, xm, A64, B64, alpha)
    rs = ref["active"][0]
    diff = np.setxor1d(gs, rs)
    if diff.size:
        bias = np.zeros(F) if layer_cpu.get("b_gate") is None else np.abs(layer_cpu["b_gate"].double().numpy())
        xa = np.abs(xm.to_f64()[0])
        pmag = np.abs(A64) @ (np.abs(B64) @ xa) + bias
        near_p = np.abs(ref["p"][0][diff] + alpha) <= P_BAND * pmag[diff]
        ex = ref["exact"]
        near_g = np.abs(ex["g"][0][diff]) <= TIE_REL * ex["cond"][0][diff]
        ok = near_p | near_g
        assert ok.all(), f"set differences outside the rounding bands: {diff[~ok][:8]}"
        assert diff.size <= max_exempt, f"{diff.size} neurons differ inside the bands (limit {max_exempt})"
    # the output on the GPU's own set
    gi = np.zeros((1, F), np.int32)
    gi[0, : gs.size] = gs
    want = O.decode(ffn, xm, O.EXACT, given_idx=gi, given_n=np.array([gs.size], np.int32))["out"]
    check_outputs(out.float().cpu().numpy().astype(np.float64), want, TOL[layer_cpu["wdtype"]])
    return gs, rs, out, ref


@pytest.mark.parametrize("frac", [0.1, 0.3, 0.6])
def test_svd_predictor_small_bf16(S, frac):
    layer = W.make_ffn_layer(2, seed=41, d_model=256, d_ff=1024)
    A, B = _svd_factors(layer, 16)
    xs = W.make_tokens(2, 3, seed=41, d_model=256)
    for t in range(3):
        x = xs[t:t + 1]
        alpha = _alpha_for(layer, x, A, B, frac)
        gs, rs, _, ref = run_and_check(S, layer, x, A, B, alpha)
        assert ref["candidates"][0].size > 0


def test_fp32_weights_ragged_shapes(S):
    # fp32 weights, d_ff not a multiple of the chunk, d_model of 24 bf16-units,
    # a rank that is not a multiple of the warp width
    layer = W.make_ffn_layer(1, seed=43, d_model=96, d_ff=701)
    x = W.make_tokens(1, 1, seed=43, d_model=96)
    A, B = _random_factors(701, 96, 13, seed=43, x=x)
    alpha = _alpha_for(layer, x, A, B, 0.4)
    run_and_check(S, layer, x, A, B, alpha)


def test_bf16_ragged_model_width(S):
    layer = W.make_ffn_layer(2, seed=44, d_model=200, d_ff=333)
    x = W.make_tokens(2, 1, seed=44, d_model=200)
    A, B = _random_factors(333, 200, 40, seed=44, x=x)
    run_and_check(S, layer, x, A, B, _alpha_for(layer, x, A, B, 0.35))


def test_infinite_alpha_is_the_exact_decode(S):
    layer = W.make_ffn_layer(2, seed=45, d_model=256, d_ff=1024)
    x = W.make_tokens(2, 1, seed=45, d_model=256)
    gs, rs, out, _ = run_and_check(S, layer, x, None, None, float("inf"))
    # the same set as sffn_decode's exact rule
    w = S.Weights(layer_to(layer, "cuda"))
    o2, i2, n2 = S.decode(x.cuda(), w, S.MODE_EXACT)
    torch.cuda.synchronize()
    assert np.array_equal(gs, i2[0, : int(n2.item())].cpu().numpy())


def test_boundary_and_empty_candidate_sets(S):
    # A = 0 and a constant bias of -1: every p_j is exactly -1
    layer = W.make_ffn_layer(1, seed=46, d_model=64, d_ff=300)
    F, d = 300, 64
    A = np.zeros((F, 8), np.float32)
    B = np.ones((8, d), np.float32)
    x = W.make_tokens(1, 1, seed=46, d_model=64)
    # alpha = 1: p_j = -1 >= -1 for every j -> the exact decode's set
    gs, rs, _, ref = run_and_check(S, layer, x, A, B, 1.0)
    assert ref["candidates"][0].size == F
    ex = O.decode(ffn_from_layer(layer), mat_from_act(x), O.EXACT)
    assert np.array_equal(rs, ex["active_idx"][0, : ex["n_active"][0]])
    # alpha = 0.5: no candidate, a zero output
    gs, rs, out, ref = run_and_check(S, layer, x, A, B, 0.5)
    assert gs.size == 0 and rs.size == 0 and not out.float().abs().sum().item()


def test_llama_shape_random_factors(S):
    # the decode workload's layer shape (d_model 4096, d_ff 11008, bf16 ReGLU),
    # random rank-256 factors: about a quarter of the neurons are candidates
    c = W.CONFIGS[2]
    layer = W.make_ffn_layer(2, seed=47)
    xs = W.make_tokens(2, 2, seed=47)
    A, B = _random_factors(c["d_ff"], c["d_model"], 256, seed=47, x=xs[:1])
    for t in range(2):
        x = xs[t:t + 1]
        run_and_check(S, layer, x, A, B, _alpha_for(layer, x, A, B, 0.25))
