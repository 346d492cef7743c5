"""GPU parity of sffn_decode against the fp64 oracle (sets within the tie band,
outputs within the per-token relative L2 bound), through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.parity import run_and_check_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    from activation_sparse_ffn_gemv_gb300 import sffn as S
    S.lib()
    return S


def _cfg(base, **kw):
    c = dict(W.CONFIGS[base])
    c.update(kw)
    return c


# small shapes: several gate chunks, ragged tails (d not a multiple of 256, F not
# a multiple of the chunk), both weight dtypes, 1..8 tokens
SMALL = [
    # (cfg, d, F, wdtype, act, B)
    (1, 256, 688, "f32", "relu", 1),
    (1, 136, 1001, "f32", "relu", 3),
    (2, 520, 1333, "bf16", "relu", 1),
    (2, 264, 777, "bf16", "relu", 2),
    (2, 1024, 2050, "bf16", "relu", 5),
    (2, 4096, 300, "bf16", "relu", 8),
    (2, 8, 33, "bf16", "relu", 1),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_exact_gating_small(sffn, case):
    cfg, d, F, wd, act, B = case
    layer = W.make_ffn_layer(cfg, seed=7, d_model=d, d_ff=F, wdtype=wd, act=act)
    x = W.make_tokens(cfg, B, seed=3, d_model=d, xdtype="f32" if wd == "f32" else "bf16")
    r = run_and_check_decode(sffn, layer, x, "exact")
    assert (r["n_active"] > 0).all()


@pytest.mark.parametrize("score", ["gate", "gate_up"])
@pytest.mark.parametrize("B", [1, 4])
def test_threshold_small(sffn, score, B):
    d, F = 512, 1536
    layer = W.make_ffn_layer(3, seed=11, d_model=d, d_ff=F)
    x = W.make_tokens(3, B, seed=5, d_model=d)
    # tau at a mid quantile of the oracle's own scores so the set is non-trivial
    from tests.oracle_io import ffn_from_layer, mat_from_act
    import oracle as O
    ref = O.decode(ffn_from_layer(layer), mat_from_act(x), O.THRESHOLD,
                   O.SCORE_GATE if score == "gate" else O.SCORE_GATE_UP, 0.0, details=True)
    tau = float(np.quantile(ref["score"], 0.7))
    r = run_and_check_decode(sffn, layer, x, "threshold", score, tau)
    frac = r["n_active"].mean() / F
    assert 0.2 < frac < 0.4


@pytest.mark.parametrize("score", ["gate", "gate_up"])
@pytest.mark.parametrize("ratio", [1.0, 0.5, 0.25, 0.125, 1e-6])
def test_keep_ratio_small(sffn, score, ratio):
    d, F = 384, 1100
    layer = W.make_ffn_layer(3, seed=13, d_model=d, d_ff=F)
    x = W.make_tokens(3, 2, seed=6, d_model=d)
    run_and_check_decode(sffn, layer, x, "keep_ratio", score, ratio)


def test_keep_ratio_batch_union(sffn):
    d, F = 256, 700
    layer = W.make_ffn_layer(3, seed=17, d_model=d, d_ff=F)
    x = W.make_tokens(3, 7, seed=8, d_model=d)
    run_and_check_decode(sffn, layer, x, "keep_ratio", "gate", 0.3)


def test_threshold_zero_is_dense(sffn):
    d, F = 256, 640
    layer = W.make_ffn_layer(3, seed=19, d_model=d, d_ff=F)
    x = W.make_tokens(3, 3, seed=9, d_model=d)
    r = run_and_check_decode(sffn, layer, x, "threshold", "gate", 0.0)
    assert (r["n_active"] == F).all()


def test_no_active_neuron_gives_zero(sffn):
    d, F = 64, 100
    layer = W.make_ffn_layer(2, seed=23, d_model=d, d_ff=F)
    layer["b_gate"] = torch.full((F,), -1e4)
    x = W.make_tokens(2, 2, seed=1, d_model=d)
    r = run_and_check_decode(sffn, layer, x, "exact")
    assert (r["n_active"] == 0).all()
    assert not torch.any(r["out"].float() != 0)


def test_ties_keep_lower_index(sffn):
    # duplicated neurons have bit-identical scores; keep-ratio must take the lower index
    d, F = 64, 64
    layer = W.make_ffn_layer(3, seed=29, d_model=d, d_ff=F)
    for name in ("w_gate", "w_up", "w_downT"):
        layer[name][32:] = layer[name][:32]
    x = W.make_tokens(3, 1, seed=2, d_model=d)
    r = run_and_check_decode(sffn, layer, x, "keep_ratio", "gate", 0.25)
    assert r["exempt"] == 0


# full configuration shapes (a few tokens; the oracle computes them one by one)

def test_config_tiny_reglu_full(sffn):
    layer = W.make_ffn_layer(1, seed=0)
    x = W.make_tokens(1, 64, seed=0)
    r = run_and_check_decode(sffn, layer, x, "exact", batch=1)
    assert abs(r["n_active"].mean() / layer["d_ff"] - 0.1587) < 0.01


@pytest.mark.parametrize("B", [1, 8])
def test_config_llama_reglu_full(sffn, B):
    layer = W.make_ffn_layer(2, seed=0)
    x = W.make_tokens(2, B, seed=B)
    r = run_and_check_decode(sffn, layer, x, "exact", nthreads=16)
    assert abs(r["n_active"].mean() / layer["d_ff"] - 0.125) < 0.02


@pytest.mark.parametrize("M", [1, 2, 4, 8])
def test_config_qwen_keep_ratio_full(sffn, M):
    layer = W.make_ffn_layer(3, seed=0, layer=M)
    x = W.make_tokens(3, 1, seed=M)
    run_and_check_decode(sffn, layer, x, "keep_ratio", "gate_up", 1.0 / M, nthreads=16)


# int4 group-quantised weights (symmetric codes, fp16 scale per 64 columns)

def _tau_at(layer, x, q, score="gate"):
    from tests.oracle_io import ffn_from_layer, mat_from_act
    import oracle as O
    ref = O.decode(ffn_from_layer(layer), mat_from_act(x), O.THRESHOLD,
                   O.SCORE_GATE if score == "gate" else O.SCORE_GATE_UP, 0.0, details=True, nthreads=16)
    return float(np.quantile(ref["score"], q))


@pytest.mark.parametrize("case", [(512, 700, 1), (1024, 2050, 3), (512, 96, 8)], ids=lambda c: "-".join(map(str, c)))
@pytest.mark.parametrize("score", ["gate", "gate_up"])
def test_int4_threshold_small(sffn, case, score):
    d, F, B = case
    layer = W.make_ffn_layer(4, seed=31, d_model=d, d_ff=F)
    x = W.make_tokens(4, B, seed=7, d_model=d)
    tau = _tau_at(layer, x, 0.8, score)
    r = run_and_check_decode(sffn, layer, x, "threshold", score, tau)
    assert 0.1 < r["n_active"].mean() / F < 0.3


def test_int4_exact_silu_is_dense(sffn):
    # SiLU is almost never exactly 0: exact gating keeps (nearly) every neuron
    d, F = 512, 300
    layer = W.make_ffn_layer(4, seed=33, d_model=d, d_ff=F)
    x = W.make_tokens(4, 2, seed=8, d_model=d)
    r = run_and_check_decode(sffn, layer, x, "exact")
    assert (r["n_active"] >= F - 2).all()


@pytest.mark.parametrize("a", [0.1, 0.6])
def test_config_qwen_int4_threshold_full(sffn, a):
    layer = W.make_ffn_layer(4, seed=0, layer=int(a * 10))
    x = W.make_tokens(4, 1, seed=int(a * 10))
    tau = _tau_at(layer, x, 1.0 - a)
    r = run_and_check_decode(sffn, layer, x, "threshold", "gate", tau, nthreads=16)
    assert abs(r["n_active"].mean() / layer["d_ff"] - a) < 0.01


@pytest.mark.parametrize("score", ["gate", "gate_up"])
@pytest.mark.parametrize("B", [1, 4])
def test_int4_keep_ratio(sffn, score, B):
    # int4-g64 weights in the keep-ratio path: scores from the int4 gate
    # kernel, the radix select, then the scaled int4 W_up / W_downT rows
    layer = W.make_ffn_layer(4, seed=11, d_model=512, d_ff=1024)
    x = W.make_tokens(4, 2 * B, seed=11, d_model=512)
    run_and_check_decode(sffn, layer, x, "keep_ratio", score, 0.125, batch=B)


def test_int4_keep_ratio_config_shape(sffn):
    # the int4 workload's layer shape (d_model 2048, d_ff 11008), tier M = 4
    layer = W.make_ffn_layer(4, seed=12)
    x = W.make_tokens(4, 2, seed=12)
    run_and_check_decode(sffn, layer, x, "keep_ratio", "gate_up", 0.25, batch=1, nthreads=16)


# More neurons than (#SMs x 256): the gate kernel's chunks cannot all be resident
# at once, so the lists and output slices are formed by a separate kernel.
BIG_F = [
    # (cfg, d, F, wdtype, mode, score, B)
    (2, 64, 40000, "bf16", "exact", "gate", 1),
    (2, 72, 39001, "bf16", "exact", "gate", 3),
    (1, 32, 40960, "f32", "threshold", "gate_up", 2),
    (4, 512, 40000, "int4_g64", "threshold", "gate", 1),
    (3, 64, 40000, "bf16", "keep_ratio", "gate_up", 1),  # scores beyond the shared-memory stage
    (3, 64, 40000, "bf16", "keep_ratio", "gate", 2),
]


@pytest.mark.parametrize("case", BIG_F, ids=lambda c: "-".join(map(str, c)))
def test_more_chunks_than_sms(sffn, case):
    cfg, d, F, wd, mode, score, B = case
    layer = W.make_ffn_layer(cfg, seed=41, d_model=d, d_ff=F, wdtype=wd,
                             act="silu" if wd == "int4_g64" else "relu")
    x = W.make_tokens(cfg, B, seed=9, d_model=d, xdtype="f32" if wd == "f32" else "bf16")
    param = {"threshold": lambda: _tau_at(layer, x, 0.85, score), "keep_ratio": lambda: 0.125,
             "exact": lambda: 0.0}[mode]()
    r = run_and_check_decode(sffn, layer, x, mode, score, param, nthreads=16)
    assert (r["n_active"] > 0).all()


# Limits of the boundary: one neuron, and the largest d_ff (65536) the decode
# call accepts (256 chunks of 256 neurons: the unfused finish).
EDGE = [
    (2, 64, 1, "bf16", "exact", "gate", 1),
    (2, 8, 1, "bf16", "exact", "gate", 8),
    (2, 64, 65536, "bf16", "exact", "gate", 2),
    (3, 64, 65536, "bf16", "keep_ratio", "gate", 1),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "-".join(map(str, c)))
def test_edge_shapes(sffn, case):
    cfg, d, F, wd, mode, score, B = case
    layer = W.make_ffn_layer(cfg, seed=43, d_model=d, d_ff=F, wdtype=wd)
    if F == 1:
        layer["b_gate"] = torch.full((1,), 2.0)  # the single neuron is active for most tokens
    x = W.make_tokens(cfg, B, seed=11, d_model=d)
    param = 0.125 if mode == "keep_ratio" else 0.0
    r = run_and_check_decode(sffn, layer, x, mode, score, param, nthreads=16)
    if mode == "keep_ratio":
        assert (r["n_active"] == max(1, int(F * param))).all()


# The tensor-core path (int4 at any token count, bf16 with 2..8 tokens) at the
# full configuration shapes, and the dense layer (every neuron) it is measured
# against.

@pytest.mark.parametrize("B", [2, 4, 8])
def test_config_qwen_int4_threshold_batched(sffn, B):
    layer = W.make_ffn_layer(4, seed=0, layer=20 + B)
    x = W.make_tokens(4, B, seed=20 + B)
    tau = _tau_at(layer, x, 0.9)
    r = run_and_check_decode(sffn, layer, x, "threshold", "gate", tau, nthreads=16)
    assert abs(r["n_active"].mean() / layer["d_ff"] - 0.1) < 0.02


@pytest.mark.parametrize("B", [2, 4])
def test_config_llama_reglu_batched(sffn, B):
    layer = W.make_ffn_layer(2, seed=0, layer=B)
    x = W.make_tokens(2, B, seed=30 + B)
    r = run_and_check_decode(sffn, layer, x, "exact", nthreads=16)
    assert abs(r["n_active"].mean() / layer["d_ff"] - 0.125) < 0.02


@pytest.mark.parametrize("d,F,mode", [(1024, 1500, "exact"), (4096, 2900, "threshold"), (512, 37, "threshold"),
                                      (2048, 40, "exact"), (4096, 11008, "exact")])
def test_int4_single_token_shapes(sffn, d, F, mode):
    # one token with int4 weights at each supported d_model: ReLU + bias for
    # exact gating, SiLU with a threshold at the 0.7 quantile; ragged chunks
    act = "relu" if mode == "exact" else "silu"
    layer = W.make_ffn_layer(4, seed=41 + d + F, d_model=d, d_ff=F, act=act)
    if mode == "exact":
        layer["b_gate"] = torch.full((F,), -0.05)
    x = W.make_tokens(4, 1, seed=41 + F, d_model=d)
    if mode == "exact":
        r = run_and_check_decode(sffn, layer, x, "exact")
    else:
        r = run_and_check_decode(sffn, layer, x, "threshold", "gate", _tau_at(layer, x, 0.7))
    assert 0 < r["n_active"][0] < F


def test_int4_exact_relu_small_chunks(sffn):
    # int4 weights with ReLU gating and a bias; ragged last tile of each chunk
    d, F = 1024, 1500
    layer = W.make_ffn_layer(4, seed=35, d_model=d, d_ff=F, act="relu")
    layer["b_gate"] = torch.full((F,), -0.05)
    x = W.make_tokens(4, 3, seed=35, d_model=d)
    r = run_and_check_decode(sffn, layer, x, "exact")
    assert (r["n_active"] > 0).all() and (r["n_active"] < F).all()


DENSE = [
    # (cfg, d, F, wdtype, act, B)
    (4, 2048, 11008, "int4_g64", "silu", 1),
    (4, 4096, 3000, "int4_g64", "silu", 1),
    (4, 512, 333, "int4_g64", "relu", 1),
    (4, 1024, 700, "int4_g64", "silu", 1),
    (4, 1024, 700, "int4_g64", "silu", 3),
    (2, 4096, 11008, "bf16", "relu", 1),
    (3, 1024, 2050, "bf16", "silu", 8),
]


@pytest.mark.parametrize("case", DENSE, ids=lambda c: "-".join(map(str, c)))
def test_dense_layer_matches_oracle(sffn, case):
    from tests.oracle_io import ffn_from_layer, mat_from_act
    from tests.parity import TOL, check_outputs, layer_to
    import oracle as O
    cfg, d, F, wd, act, B = case
    layer = W.make_ffn_layer(cfg, seed=71, d_model=d, d_ff=F, wdtype=wd, act=act)
    x = W.make_tokens(cfg, B, seed=71, d_model=d)
    w = sffn.Weights(layer_to(layer, "cuda"))
    out = sffn.decode_dense(x.cuda(), w)
    torch.cuda.synchronize()
    # threshold 0 on the gate score keeps every neuron: the dense FFN (pinned)
    ref = O.decode(ffn_from_layer(layer), mat_from_act(x), O.THRESHOLD, O.SCORE_GATE, 0.0, nthreads=16)
    assert (ref["n_active"] == F).all()
    check_outputs(out.float().cpu().numpy().astype(np.float64), ref["out"], TOL[wd])


# sffn_gate_scores: the per-neuron scores themselves against the oracle's, within
# 1e-5 of the oracle's bound on the score computation (cond).  One token with
# int4 weights and the gate-and-up score runs the int4 score stream; the other
# cases the gate kernel.
@pytest.mark.parametrize("cfg,wd,B", [(4, "int4_g64", 1), (4, "int4_g64", 3), (3, "bf16", 1)],
                         ids=["int4-B1", "int4-B3", "bf16-B1"])
@pytest.mark.parametrize("score", ["gate", "gate_up"])
def test_gate_scores_match_the_oracle(sffn, cfg, wd, B, score):
    from tests.oracle_io import ffn_from_layer, mat_from_act
    from tests.parity import layer_to
    import oracle as O
    d, F = 1024, 1500
    layer = W.make_ffn_layer(cfg, seed=57, d_model=d, d_ff=F, wdtype=wd)
    x = W.make_tokens(cfg, B, seed=57, d_model=d)
    w = sffn.Weights(layer_to(layer, "cuda"))
    w.set_down_norms(sffn.down_norms(w))
    kind = sffn.SCORE_GATE if score == "gate" else sffn.SCORE_GATE_UP
    sc = sffn.gate_scores(x.cuda(), w, kind)
    torch.cuda.synchronize()
    ref = O.decode(ffn_from_layer(layer), mat_from_act(x), O.THRESHOLD,
                   O.SCORE_GATE if score == "gate" else O.SCORE_GATE_UP, 0.0, details=True, nthreads=8)
    got = sc.cpu().numpy().astype(np.float64)
    err = np.abs(got - ref["score"])
    bound = 1e-5 * ref["cond"] + 1e-12
    assert (err <= bound).all(), f"max err / cond {np.max(err / (ref['cond'] + 1e-30)):.3e}"
    assert np.all(got >= 0.0)
