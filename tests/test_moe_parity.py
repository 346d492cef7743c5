"""GPU parity of the MoE routing and block budget against the fp64 oracle
(oracle/moe.py), plus the host-side schedule and argument checks (CPU).

* sffn_moe_route: K, the ascending experts and the renormalised weights per
  token.  The GPU decides the bucket in fp32: a token whose top-b mass for some
  admissible bucket b lies within 1e-5 of the threshold may take the neighbouring
  bucket and is exempt (at most 2 per call); every other token is exact, and its
  weights agree to 1e-5 relative.
* sffn_moe_block_budget: the chosen blocks, the token list and the ranges.  The
  blocks are exact except where two blocks' summed importances lie within 1e-5
  (relative) of each other at the cut; the token list is the chosen blocks'
  tokens and the ranges are the list's maximal contiguous runs, exactly.
"""
from __future__ import annotations

import json
import math
import os
import ctypes as C

import numpy as np
import pytest
import torch

import oracle as O
from oracle import moe as M
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import mat_from_act

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "moe_schedule.json")
MASS_BAND = 1e-5


@pytest.fixture(scope="module")
def S():
    from activation_sparse_ffn_gemv_gb300 import build as B
    B.build()
    from activation_sparse_ffn_gemv_gb300 import sffn
    sffn.lib()
    return sffn


def test_progressive_schedule_matches_the_page_and_oracle(S):
    g = json.load(open(GOLDEN))
    for row in g["progressive"]:
        lo, hi = row["layers"]
        for layer in range(lo, hi + 1):
            assert S.moe_progressive_k(layer) == row["k"], row["cite"]
    for layer in range(0, 100):
        assert S.moe_progressive_k(layer) == M.progressive_k(layer)
    assert S.moe_progressive_k(-1) == -1


def test_route_and_budget_argument_checks(S):
    L = S.lib()
    bk = (C.c_int32 * 4)(3, 4, 5, 6)
    bad = (C.c_int32 * 2)(4, 3)

    def route(logits=16, T=4, E=16, cap=4, mass=0.5, b=bk, nb=4, kmax=4, ko=16, ex=16, wt=16):
        return L.sffn_moe_route(logits, T, E, cap, mass, b, nb, kmax, ko, ex, wt, None)

    assert route(logits=None) == S.ERR_INVALID_ARG
    assert route(ko=None) == S.ERR_INVALID_ARG
    assert route(b=None) == S.ERR_INVALID_ARG
    assert route(E=0) == S.ERR_SHAPE
    assert route(E=513) == S.ERR_SHAPE
    assert route(cap=0) == S.ERR_SHAPE
    assert route(cap=9, kmax=9) == S.ERR_SHAPE
    assert route(cap=17) == S.ERR_SHAPE            # cap <= E
    assert route(kmax=3) == S.ERR_SHAPE            # kmax >= cap
    assert route(nb=0) == S.ERR_INVALID_ARG
    assert route(b=bad, nb=2) == S.ERR_INVALID_ARG  # buckets ascending
    assert route(mass=float("nan")) == S.ERR_INVALID_ARG

    def budget(y=16, Lq=1000, d=64, mass=0.5, lo=0.1, hi=0.5, block=128, ti=16, nt=16, rg=16, nr=16):
        return L.sffn_moe_block_budget(y, Lq, d, mass, lo, hi, block, ti, nt, rg, nr, 256, 1 << 20, None)

    assert budget(y=None) == S.ERR_INVALID_ARG
    assert budget(rg=None) == S.ERR_INVALID_ARG
    assert budget(Lq=0) == S.ERR_SHAPE
    assert budget(d=12) == S.ERR_SHAPE
    assert budget(block=0) == S.ERR_SHAPE
    assert budget(Lq=1 << 20, block=64) == S.ERR_SHAPE   # more than 8192 blocks
    assert budget(lo=0.6, hi=0.5) == S.ERR_INVALID_ARG
    assert budget(hi=1.5) == S.ERR_INVALID_ARG
    assert budget(y=8) == S.ERR_ALIGNMENT
    assert L.sffn_moe_budget_workspace_size(0, 64) == 0
    assert L.sffn_moe_budget_workspace_size(1000, 64) > 0


def _logits(T, E, seed, scale=None, quant=None):
    """Router logits; by default each token has its own spread (from nearly
    flat to peaked), so every bucket occurs."""
    g = np.random.default_rng(seed)
    sc = g.uniform(1.0, 5.0, size=(T, 1)) if scale is None else scale
    z = g.standard_normal((T, E)) * sc
    if quant:
        z = np.round(z / quant) * quant
    return z.astype(np.float32)


def check_route(S, z, layer, mass=0.5, buckets=M.BUCKETS, max_exempt=2):
    cap = M.progressive_k(layer)
    k, ex, wt = S.moe_route(torch.from_numpy(z).cuda(), cap, mass, buckets)
    torch.cuda.synchronize()
    k, ex, wt = k.cpu().numpy(), ex.cpu().numpy(), wt.cpu().numpy()
    ref = M.route(z.astype(np.float64), layer, mass, buckets)
    P = M.softmax(z.astype(np.float64))
    exempt = 0
    for t, (rk, rex, rw) in enumerate(ref):
        order = M.expert_order(P[t])
        near = any(b <= cap and abs(P[t][order[:b]].sum() - mass) <= MASS_BAND for b in buckets)
        if k[t] != rk:
            assert near, f"token {t}: K {k[t]} vs {rk} away from the mass threshold"
            exempt += 1
            continue
        assert np.array_equal(ex[t, :rk], rex) and np.all(ex[t, rk:] == -1), (t, ex[t], rex)
        np.testing.assert_allclose(wt[t, :rk], rw, rtol=1e-5, atol=1e-7)
        assert np.all(wt[t, rk:] == 0)
    assert exempt <= max_exempt
    return k


@pytest.mark.gpu
@pytest.mark.parametrize("E", [16, 100, 384, 512])
@pytest.mark.parametrize("layer", [3, 20, 45])
def test_route_matches_the_oracle(S, E, layer):
    z = _logits(256, E, seed=E + layer)
    k = check_route(S, z, layer)
    assert len(set(k.tolist())) > 1   # more than one bucket occurs


@pytest.mark.gpu
def test_route_ties_and_custom_buckets(S):
    z = _logits(128, 64, seed=5, quant=0.5)          # many equal logits: ties to the lower expert
    check_route(S, z, 3)
    check_route(S, _logits(128, 64, seed=6), 3, mass=0.3, buckets=(2, 5))
    u = np.zeros((8, 16), np.float32)                # uniform: top-6 holds 6/16 < 0.5 -> K = cap
    k = check_route(S, u, 3)
    assert np.all(k == 6)


def check_budget(S, ya_cpu, mass, lo=0.10, hi=0.50, block=128):
    L = ya_cpu.shape[0]
    ti, nt, rg, nr = S.moe_block_budget(ya_cpu.cuda(), mass, lo, hi, block)
    torch.cuda.synchronize()
    n, nrg = int(nt.item()), int(nr.item())
    got = ti[:n].cpu().numpy()
    rgs = [tuple(r) for r in rg[:nrg].cpu().numpy().tolist()]
    assert rgs == M.ranges(got)                      # ranges: the list's maximal runs
    assert np.all(np.diff(got) > 0)
    s = O.token_norms(mat_from_act(ya_cpu))
    want = M.block_budget(s, mass, lo, hi, block)
    nblocks = (L + block - 1) // block
    gb = sorted(set((got // block).tolist()))
    wb = sorted(set((want // block).tolist()))
    # every chosen block is whole
    assert n == sum(min(L, (b + 1) * block) - b * block for b in gb)
    if gb != wb:
        bsum = np.array([s[i * block:(i + 1) * block].sum() for i in range(nblocks)])
        d = sorted(set(gb) ^ set(wb))
        if len(gb) == len(wb):
            cut = bsum[wb].min()
            assert all(abs(bsum[b] - cut) <= MASS_BAND * cut for b in d), (d, bsum[d], cut)
        else:
            # the count differs only when the mass rule's prefix sits at a bucket edge
            f = M.mass_fraction(s, mass)
            edge = abs(min(max(f, lo), hi) * nblocks - round(min(max(f, lo), hi) * nblocks)) <= nblocks / L + 1e-9
            assert edge and abs(len(gb) - len(wb)) == 1
    return got, rgs


@pytest.mark.gpu
@pytest.mark.parametrize("L", [100, 128, 1000, 5000, 16384])
@pytest.mark.parametrize("mass", [0.0, 0.2, 0.5, 0.9, 1.0])
def test_block_budget_matches_the_oracle(S, L, mass):
    _, ya = W.make_prefill_inputs(L, 64, seed=L + int(mass * 10))
    check_budget(S, ya, mass)


@pytest.mark.gpu
def test_block_budget_ratios_and_block_sizes(S):
    _, ya = W.make_prefill_inputs(3000, 64, seed=17)
    for lo, hi, block in ((0.0, 1.0, 128), (0.3, 0.3, 100), (0.1, 0.5, 1), (0.1, 0.5, 3000), (0.05, 0.2, 64)):
        check_budget(S, ya, 0.5, lo, hi, block)


@pytest.mark.gpu
def test_block_budget_feeds_the_prefill(S):
    # the budget's device list drives sffn_prefill with no host round trip; the
    # result equals the prefill on the oracle's list (when the two lists agree)
    c = W.CONFIGS[5]
    L, d, F = 2048, 256, 512
    layer = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in W.make_ffn_layer(5, seed=3, d_model=d, d_ff=F).items()}
    w = S.Weights(layer)
    X, Ya = W.make_prefill_inputs(L, d, seed=3)
    X, Ya = X.cuda(), Ya.cuda()
    ti, nt, _, _ = S.moe_block_budget(Ya, 0.3)
    out = S.prefill(X, Ya, w, ti, nt)
    s = O.token_norms(mat_from_act(Ya.cpu()))
    want = M.block_budget(s, 0.3)
    torch.cuda.synchronize()
    got = ti[: int(nt.item())].cpu().numpy()
    assert np.array_equal(got, want)
    ref = S.prefill(X, Ya, w, torch.from_numpy(want).cuda(), torch.tensor([want.size], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
