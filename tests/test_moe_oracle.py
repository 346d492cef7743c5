"""Pins of the MoE top-K / block-budget oracle (oracle/moe.py), CPU."""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import pytest

from oracle import moe as M

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "moe_schedule.json")


def test_schedule_and_defaults_match_the_page():
    g = json.load(open(GOLDEN))
    for row in g["progressive"]:
        lo, hi = row["layers"]
        for layer in (lo, (lo + hi) // 2, hi):
            assert M.progressive_k(layer) == row["k"], row["cite"]
    assert M.progressive_k(61) == 4            # past the table: the last range's K
    assert list(M.BUCKETS) == g["buckets"]
    assert M.block_budget.__defaults__[:3] == (g["min_full_ratio"], g["max_full_ratio"], g["block"])


def test_bucket_closed_cases():
    # a dominant expert: the top 3 already hold half the mass
    p = np.array([0.45, 0.1, 0.1] + [0.35 / 13] * 13)
    assert M.adaptive_k(p) == 3
    # uniform over 16 experts: top-6 mass is 6/16 < 0.5 -> the largest bucket (or the cap)
    u = np.full(16, 1 / 16)
    assert M.adaptive_k(u) == 6
    assert M.adaptive_k(u, cap=4) == 4
    # exactly reaching the mass at 4 experts
    q = np.array([0.2, 0.1, 0.1, 0.1] + [0.5 / 12] * 12)
    assert M.adaptive_k(q) == 4
    # the cap limits the buckets: a token needing 5 in a deep layer (cap 4) gets 4
    r = np.array([0.12] * 4 + [0.03] * 4 + [0.4 / 20] * 20)
    assert M.adaptive_k(r) == 5 and M.adaptive_k(r, cap=4) == 4


def test_route_brute_force():
    rng = np.random.default_rng(0)
    E = 10
    for layer in (3, 20, 45):
        logits = rng.normal(size=(6, E)) * 1.5
        P = M.softmax(logits)
        for t, (k, experts, w) in enumerate(M.route(logits, layer)):
            assert k <= M.progressive_k(layer) and k in set(M.BUCKETS) | {M.progressive_k(layer)}
            # the chosen set maximises the kept probability among size-k sets
            best = max(itertools.combinations(range(E), k), key=lambda c: (P[t, list(c)].sum(), [-i for i in c]))
            assert experts.tolist() == sorted(best)
            assert w.sum() == pytest.approx(1.0) and np.all(np.diff(experts) > 0)
            # the smallest admissible bucket: any smaller bucket misses the mass
            for b in M.BUCKETS:
                if b < k:
                    assert np.sort(P[t])[::-1][:b].sum() < 0.5


def test_block_budget_brute_force():
    rng = np.random.default_rng(1)
    block = 4
    for trial in range(20):
        L = int(rng.integers(1, 7)) * block + int(rng.integers(0, block))
        s = rng.random(L) * np.exp(rng.normal(size=L))
        mass = float(rng.choice([0.0, 0.2, 0.5, 0.9, 1.0]))
        sel = M.block_budget(s, mass, 0.1, 0.5, block)
        nblocks = math.ceil(L / block)
        f = min(max(M.mass_fraction(s, mass), 0.1), 0.5)
        nsel = max(1, min(nblocks, math.ceil(f * nblocks - 1e-12)))
        bsum = [s[i * block:(i + 1) * block].sum() for i in range(nblocks)]
        best = max(itertools.combinations(range(nblocks), nsel),
                   key=lambda c: (sum(bsum[i] for i in c), [-i for i in c]))
        want = np.concatenate([np.arange(b * block, min(L, (b + 1) * block)) for b in sorted(best)])
        assert sel.tolist() == want.tolist()
        # whole blocks: few contiguous ranges
        assert len(M.ranges(sel)) <= nsel


def test_mass_fraction_cases():
    s = np.array([4.0, 1.0, 3.0, 2.0])          # total 10
    assert M.mass_fraction(s, 0.4) == 0.25       # 4 >= 4
    assert M.mass_fraction(s, 0.5) == 0.5        # 4 + 3 >= 5
    assert M.mass_fraction(s, 1.0) == 1.0
    assert M.mass_fraction(s, 0.0) == 0.0
    assert M.mass_fraction(np.zeros(5), 0.3) == 1.0   # all-zero importance: every token
    assert M.ranges(np.array([0, 1, 2, 5, 6, 9])) == [(0, 3), (5, 7), (9, 10)]
