"""GPU parity of the keep-ratio tier tables against the fp64 oracle
(oracle/tiers.py).

* sffn_tier_core_set is integer and index work on given scores: bit-exact
  against core_set on the same fp32 scores (ties in scores and in counts go to
  the lower index on both sides).
* sffn_decode_tiered: the kept set is core U the largest scores outside the
  core.  It is compared with select_with_core on the oracle's fp64 scores,
  bit-exact except for columns within the decode's tie band of the cut (at most
  two per token); the output is compared with the oracle's output on the GPU's
  own set.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from oracle import tiers as T
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import ffn_from_layer, mat_from_act
from tests.parity import TIE_REL, TOL, check_outputs, layer_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from activation_sparse_ffn_gemv_gb300 import build as B
    B.build()
    from activation_sparse_ffn_gemv_gb300 import sffn
    sffn.lib()
    return sffn


def _calib(N, F, seed, quant=None):
    g = np.random.default_rng(seed)
    s = np.abs(g.standard_normal((N, F))) * np.exp(0.7 * g.standard_normal(F))[None, :]
    if quant:
        s = np.round(s / quant) * quant   # many equal scores
    return s.astype(np.float32)


@pytest.mark.parametrize("N,F,k,c,quant", [
    (40, 1000, 100, 37, None), (40, 1000, 100, 0, None), (40, 1000, 100, 100, None), (40, 1000, 100, 150, None),
    (33, 997, 64, 50, 0.5), (16, 700, 90, 45, 10.0), (64, 11008, 1376, 688, None), (3, 50000, 400, 300, None),
    (1, 64, 64, 64, None),
])
def test_core_set_matches_the_oracle(S, N, F, k, c, quant):
    s = _calib(N, F, seed=N * 7 + F, quant=quant)
    core = S.tier_core_set(torch.from_numpy(s).cuda(), k, c)
    torch.cuda.synchronize()
    want = T.core_set(s.astype(np.float64), k, c)
    assert np.array_equal(core.cpu().numpy(), want)


def test_core_set_all_equal_scores(S):
    s = np.ones((5, 300), np.float32)
    core = S.tier_core_set(torch.from_numpy(s).cuda(), 40, 25)
    torch.cuda.synchronize()
    assert core.cpu().tolist() == list(range(25)) == T.core_set(s.astype(np.float64), 40, 25).tolist()


def run_tiered(S, layer_cpu, x_cpu, score, ratio, core_np, max_exempt=2):
    dev = "cuda"
    w = S.Weights(layer_to(layer_cpu, dev))
    w.set_down_norms(S.down_norms(w))
    x = x_cpu.to(dev)
    core = None if core_np is None else torch.from_numpy(core_np.astype(np.int32)).to(dev)
    out, idx, n = S.decode_tiered(x, w, score, ratio, core)
    torch.cuda.synchronize()
    B, F = x_cpu.shape[0], layer_cpu["d_ff"]
    idx, n = idx.cpu().numpy(), n.cpu().numpy()
    sets = [idx[b, : n[b]] for b in range(B)]
    gi = np.zeros((B, F), np.int32)
    for b, st in enumerate(sets):
        gi[b, : st.size] = st
    ffn, xm = ffn_from_layer(layer_cpu), mat_from_act(x_cpu)
    osc = O.SCORE_GATE_UP if score == S.SCORE_GATE_UP else O.SCORE_GATE
    ref = O.decode(ffn, xm, O.KEEP_RATIO, osc, ratio, given_idx=gi, given_n=n.astype(np.int32), details=True)
    k = O.keep_count(F, ratio)
    cz = np.zeros(0, np.int32) if core_np is None else core_np.astype(np.int32)
    exempt = 0
    for b in range(B):
        gs = sets[b]
        assert gs.size == 0 or (np.all(np.diff(gs) > 0) and gs[0] >= 0 and gs[-1] < F)
        want = T.select_with_core(ref["score"][b], k, cz)
        assert set(cz.tolist()) <= set(gs.tolist())
        assert gs.size == max(k, cz.size)
        diff = np.setxor1d(gs, want)
        if diff.size:
            extra = np.setdiff1d(want, cz)
            cut = ref["score"][b][extra].min()
            band = TIE_REL * np.maximum(abs(cut), ref["cond"][b][diff])
            bad = diff[np.abs(ref["score"][b][diff] - cut) > band]
            assert bad.size == 0, f"token {b}: differences outside the tie band: {bad[:6]}"
            exempt += diff.size
    assert exempt <= 2 * B, f"{exempt} columns differ inside the tie band"
    check_outputs(out.float().cpu().numpy().astype(np.float64), ref["out"], TOL[layer_cpu["wdtype"]])
    return sets, out


def _layer_and_core(S, score, F=1024, d=256, ratio=0.25, c_frac=0.5, seed=31):
    layer = W.make_ffn_layer(3, seed=seed, d_model=d, d_ff=F)
    k = O.keep_count(F, ratio)
    # calibration: the layer's own scores on 32 tokens, through the library
    w = S.Weights(layer_to(layer, "cuda"))
    w.set_down_norms(S.down_norms(w))
    xc = W.make_tokens(3, 32, seed=seed + 1, d_model=d).cuda()
    sc = torch.cat([S.gate_scores(xc[i:i + 8], w, score) for i in range(0, 32, 8)])
    core = S.tier_core_set(sc, k, int(c_frac * k))
    torch.cuda.synchronize()
    assert np.array_equal(core.cpu().numpy(), T.core_set(sc.cpu().numpy().astype(np.float64), k, int(c_frac * k)))
    return layer, core.cpu().numpy()


@pytest.mark.parametrize("score_name", ["gate", "gate_up"])
@pytest.mark.parametrize("B", [1, 4])
def test_tiered_decode_with_a_calibrated_core(S, score_name, B):
    score = S.SCORE_GATE if score_name == "gate" else S.SCORE_GATE_UP
    layer, core = _layer_and_core(S, score)
    x = W.make_tokens(3, B, seed=77, d_model=256)
    run_tiered(S, layer, x, score, 0.25, core)


def test_empty_core_is_the_keep_ratio_decode(S):
    layer = W.make_ffn_layer(3, seed=32, d_model=256, d_ff=1024)
    x = W.make_tokens(3, 2, seed=32, d_model=256)
    sets, out = run_tiered(S, layer, x, S.SCORE_GATE_UP, 0.125, None)
    w = S.Weights(layer_to(layer, "cuda"))
    w.set_down_norms(S.down_norms(w))
    o2, i2, n2 = S.decode(x.cuda(), w, S.MODE_KEEP_RATIO, S.SCORE_GATE_UP, 0.125)
    torch.cuda.synchronize()
    for b in range(2):
        assert np.array_equal(sets[b], i2[b, : int(n2[b])].cpu().numpy())
    assert torch.equal(out, o2)


def test_core_of_k_or_more_is_kept_alone(S):
    layer = W.make_ffn_layer(3, seed=33, d_model=128, d_ff=512)
    x = W.make_tokens(3, 1, seed=33, d_model=128)
    k = O.keep_count(512, 0.125)
    core = np.arange(3, 3 + 7 * k, 7)[: k]            # exactly k
    sets, _ = run_tiered(S, layer, x, S.SCORE_GATE, 0.125, core)
    assert np.array_equal(sets[0], core)
    big = np.arange(0, 512, 3)[: k + 20]              # more than k
    sets, _ = run_tiered(S, layer, x, S.SCORE_GATE, 0.125, big)
    assert np.array_equal(sets[0], big)


def test_core_index_out_of_range_is_skipped_and_reported(S):
    layer = W.make_ffn_layer(3, seed=34, d_model=128, d_ff=512)
    x = W.make_tokens(3, 1, seed=34, d_model=128).cuda()
    w = S.Weights(layer_to(layer, "cuda"))
    w.set_down_norms(S.down_norms(w))
    ws = S.alloc_workspace(S.WS_DECODE, 1, w)
    good = torch.tensor([5, 40, 300], dtype=torch.int32, device="cuda")
    bad = torch.tensor([5, 40, 300, 900], dtype=torch.int32, device="cuda")
    o1, i1, n1 = S.decode_tiered(x, w, S.SCORE_GATE, 0.125, good, workspace=ws)
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == 0
    o2, i2, n2 = S.decode_tiered(x, w, S.SCORE_GATE, 0.125, bad, workspace=ws)
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == S.ERR_DEVICE
    assert torch.equal(n1, n2) and torch.equal(i1[0, : int(n1)], i2[0, : int(n2)]) and torch.equal(o1, o2)


def test_qwen_shape_tier(S):
    # the keep-ratio workload's layer shape (d_model 2048, d_ff 11008), tier M = 8
    # with a core of half the tier from 64 calibration tokens
    layer, core = _layer_and_core(S, S.SCORE_GATE_UP, F=11008, d=2048, ratio=0.125, c_frac=0.5, seed=35)
    x = W.make_tokens(3, 2, seed=36, d_model=2048)
    run_tiered(S, layer, x, S.SCORE_GATE_UP, 0.125, core)
