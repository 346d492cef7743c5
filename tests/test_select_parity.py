"""GPU parity of sffn_token_select against the fp64 oracle: the selected set is
bit-exact except for tokens whose importance lies within 1e-6 (relative) of a
cut of the selection (the crossing value of the mass prefix or of the
min_keep extension)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import mat_from_act
from tests.parity import TIE_REL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    from activation_sparse_ffn_gemv_gb300 import sffn as S
    S.lib()
    return S


def _oracle_cuts(s, sel, pre, L, recent_n):
    """Importance values at which the oracle's selection was cut."""
    cuts = []
    if len(pre) and len(pre) < L:
        cuts.append(s[pre].min())
    tail = set(range(max(0, L - recent_n), L))
    ext = [t for t in sel.tolist() if t not in set(pre.tolist()) and t not in tail]
    if ext:
        cuts.append(s[ext].min())
    return cuts


def check_select(sffn, ya_cpu: torch.Tensor, m: float, recent_n: int, min_keep: int, max_exempt: int = 2):
    """GPU selection vs the oracle: bit-exact except tokens whose importance lies
    within the tie band of one of the oracle's cuts, at most ``max_exempt`` of them."""
    L = ya_cpu.shape[0]
    sel_g, n_g = sffn.token_select(ya_cpu.cuda(), m, recent_n, min_keep)
    torch.cuda.synchronize()
    n = int(n_g.item())
    g = sel_g[:n].cpu().numpy()
    assert n >= 1 or L == 0
    assert np.all(np.diff(g) > 0) and (n == 0 or (g[0] >= 0 and g[-1] < L))
    s = O.token_norms(mat_from_act(ya_cpu))
    sel, pre = O.mass_select(s, m, recent_n, min_keep)
    # guards hold on the GPU result itself
    assert set(range(max(0, L - recent_n), L)) <= set(g.tolist())
    assert n >= min(min_keep, L)
    diff = np.setxor1d(g, sel)
    if diff.size:
        cuts = _oracle_cuts(s, sel, pre, L, recent_n)
        ok = np.zeros(diff.size, bool)
        for c in cuts:
            ok |= np.abs(s[diff] - c) <= TIE_REL * np.maximum(c, s[diff])
        assert ok.all(), (f"{(~ok).sum()} tokens differ outside the tie band: {diff[~ok][:8]} "
                          f"s={s[diff[~ok][:8]]} cuts={cuts}")
        assert diff.size <= max_exempt, f"{diff.size} tokens differ inside the tie band (limit {max_exempt})"
    return g, sel, s


@pytest.mark.parametrize("m", [0.2, 0.5, 0.7, 1.0])
def test_config_prefill_selection_full(sffn, m):
    c = W.CONFIGS[5]
    _, ya = W.make_prefill_inputs(c["L"], c["d_model"], seed=0)
    g, sel, s = check_select(sffn, ya, m, c["recent_n"], c["min_keep"])
    if m == 1.0:
        assert g.size == c["L"]


# up to 32768 tokens the importances are staged in shared memory; 40000 takes the
# workspace path
@pytest.mark.parametrize("L", [1, 2, 7, 100, 1023, 1024, 1025, 4099, 32768, 40000])
@pytest.mark.parametrize("m", [0.0, 1e-9, 0.3, 0.9])
def test_lengths_and_thresholds(sffn, L, m):
    _, ya = W.make_prefill_inputs(L, 64, seed=L)
    check_select(sffn, ya, m, recent_n=5, min_keep=1)


def test_all_zero_is_dense(sffn):
    ya = torch.zeros(300, 64, dtype=torch.bfloat16)
    g, _, _ = check_select(sffn, ya, 0.4, recent_n=4, min_keep=1)
    assert g.tolist() == list(range(300))


def test_single_nonzero_token(sffn):
    ya = torch.zeros(500, 64, dtype=torch.bfloat16)
    ya[123, 5] = 3.0
    g, _, _ = check_select(sffn, ya, 0.5, recent_n=0, min_keep=1)
    assert g.tolist() == [123]


def test_ties_take_lower_indices(sffn):
    # identical rows: identical importances; the prefix takes the lowest indices.
    # With a norm of exactly 2 every mass sum is exact on both sides: 10 of 40.
    row = torch.zeros(1, 64, dtype=torch.bfloat16)
    row[0, 7] = 2.0
    g, sel, _ = check_select(sffn, row.repeat(40, 1), 0.25, recent_n=0, min_keep=1)
    assert g.tolist() == sel.tolist() == list(range(10))
    # A generic norm: in exact arithmetic 10 equal masses reach a quarter of 40.
    # The kernel's fixed-point sums are exact; the fp64 oracle's prefix sum may
    # round below the target and take an 11th token, a tie that check_select
    # already exempts.
    gen = torch.Generator().manual_seed(5)
    for _ in range(4):
        row = torch.randn(1, 64, generator=gen).to(torch.bfloat16)
        g, sel, _ = check_select(sffn, row.repeat(40, 1), 0.25, recent_n=0, min_keep=1)
        assert g.tolist() == list(range(10))
        assert sel.tolist() in (list(range(10)), list(range(11)))


# 5000/7000 tokens stage in shared memory; 50000/70000 run the multi-block passes
@pytest.mark.parametrize("k", [1, 10])
def test_ties_across_many_blocks(sffn, k):
    # 5000k equal importances of exactly 2 (every sum exact): a quarter of the
    # mass is the first 1250k tokens, whichever blocks they fall in
    row = torch.zeros(1, 64, dtype=torch.bfloat16)
    row[0, 3] = 2.0
    g, sel, _ = check_select(sffn, row.repeat(5000 * k, 1), 0.25, recent_n=0, min_keep=1)
    assert g.tolist() == sel.tolist() == list(range(1250 * k))
    # two values, the larger after the smaller: 4000k twos, then 3000k fours;
    # 0.7 of the mass is every four and the first 1000k twos
    ya = row.repeat(7000 * k, 1)
    ya[4000 * k:, 3] = 4.0
    g, sel, _ = check_select(sffn, ya, 0.7, recent_n=0, min_keep=1)
    assert g.tolist() == sel.tolist() == list(range(1000 * k)) + list(range(4000 * k, 7000 * k))


def test_recent_tail_longer_than_sequence(sffn):
    _, ya = W.make_prefill_inputs(50, 64, seed=3)
    g, _, _ = check_select(sffn, ya, 0.2, recent_n=128, min_keep=1)
    assert g.tolist() == list(range(50))


@pytest.mark.parametrize("min_keep", [1, 17, 500])
def test_min_keep_extension(sffn, min_keep):
    _, ya = W.make_prefill_inputs(1000, 64, seed=9)
    g, _, _ = check_select(sffn, ya, 0.0, recent_n=0, min_keep=min_keep)
    assert g.size == min_keep
    g2, _, _ = check_select(sffn, ya, 0.05, recent_n=3, min_keep=min_keep)
    assert g2.size >= min_keep
