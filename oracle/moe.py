"""Adaptive MoE expert top-K and the block token budget -- TEST INFRASTRUCTURE
(the fp64 oracle's part for them).  Only the tests may import this module.

The RedKnot write-up (bhfrc.com/news/43276, "自適應專家 Top-K") describes, for
MoE layers:

  1. a progressive top-K schedule by depth: layers 0-15 route each token to 6
     experts, layers 16-39 to 5, layers 40-60 to 4;
  2. an adaptive top-K: per token, the smallest K from the candidate buckets
     (3, 4, 5, 6) whose top-K routing probability mass reaches 0.50;
  3. a token budget between min_full_ratio 0.10 and max_full_ratio 0.50 of the
     tokens, chosen as whole 128-token blocks so that the routed rows form few
     contiguous ranges.

Read plainly (every free choice is stated):
  * routing probabilities are the softmax of the router logits (fp64); experts
    are ordered by probability descending, ties to the lower expert index;
  * a token's K is the smallest bucket b <= the layer's progressive K whose top-b
    mass is >= the mass threshold, else the layer's progressive K; layers past
    the last range keep its K;
  * the chosen experts' weights are their probabilities renormalised to sum 1;
  * the block budget: a token's importance is given (e.g. the L2 norm of its
    attention output); the fraction f of tokens that the mass rule of the
    token-selective FFN would keep is clamped to [min_full_ratio,
    max_full_ratio]; ceil(f * nblocks) blocks (at least one) with the largest
    summed importance run the MoE (ties to the lower block index).

Pinned by tests/test_moe_oracle.py: the schedule table, closed-form bucket cases,
brute force over expert subsets and over block subsets on small inputs.
"""
from __future__ import annotations

import math

import numpy as np

PROGRESSIVE = ((0, 15, 6), (16, 39, 5), (40, 60, 4))
BUCKETS = (3, 4, 5, 6)


def progressive_k(layer: int, schedule=PROGRESSIVE) -> int:
    for lo, hi, k in schedule:
        if lo <= layer <= hi:
            return k
    return schedule[-1][2] if layer > schedule[-1][1] else schedule[0][2]


def softmax(logits: np.ndarray) -> np.ndarray:
    z = np.asarray(logits, np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def expert_order(probs: np.ndarray) -> np.ndarray:
    """Expert indices by probability descending, ties to the lower index."""
    p = np.asarray(probs, np.float64)
    return np.lexsort((np.arange(p.size), -p))


def adaptive_k(probs: np.ndarray, mass: float = 0.5, buckets=BUCKETS, cap: int | None = None) -> int:
    p = np.asarray(probs, np.float64)
    order = expert_order(p)
    top = np.cumsum(p[order])
    limit = max(buckets) if cap is None else cap
    for b in sorted(buckets):
        if b > limit:
            break
        if top[b - 1] >= mass:
            return b
    return limit


def route(logits: np.ndarray, layer: int, mass: float = 0.5, buckets=BUCKETS, schedule=PROGRESSIVE):
    """Per token: (K, experts ascending, weights aligned with the experts)."""
    P = softmax(np.atleast_2d(logits))
    cap = progressive_k(layer, schedule)
    out = []
    for p in P:
        k = adaptive_k(p, mass, buckets, cap)
        chosen = expert_order(p)[:k]
        w = p[chosen] / p[chosen].sum()
        o = np.argsort(chosen)
        out.append((k, chosen[o].astype(np.int32), w[o]))
    return out


def mass_fraction(importance: np.ndarray, mass: float) -> float:
    """Fraction of tokens the mass rule keeps: the shortest prefix of tokens by
    importance descending (ties lower index) whose sum reaches mass * total."""
    s = np.asarray(importance, np.float64)
    L = s.size
    tot = s.sum()
    if L == 0:
        return 0.0
    if mass >= 1.0 or tot == 0.0:
        return 1.0
    if mass <= 0.0:
        return 0.0
    order = np.lexsort((np.arange(L), -s))
    c = np.cumsum(s[order])
    n = int(np.searchsorted(c, mass * tot, side="left")) + 1
    return min(n, L) / L


def block_budget(importance: np.ndarray, mass: float, min_ratio: float = 0.10, max_ratio: float = 0.50,
                 block: int = 128) -> np.ndarray:
    """Ascending token indices of the blocks that run the MoE."""
    s = np.asarray(importance, np.float64)
    L = s.size
    nblocks = (L + block - 1) // block
    if nblocks == 0:
        return np.zeros(0, np.int32)
    f = min(max(mass_fraction(s, mass), min_ratio), max_ratio)
    nsel = max(1, min(nblocks, math.ceil(f * nblocks - 1e-12)))
    bsum = np.array([s[i * block:(i + 1) * block].sum() for i in range(nblocks)])
    order = np.lexsort((np.arange(nblocks), -bsum))
    chosen = np.sort(order[:nsel])
    return np.concatenate([np.arange(b * block, min(L, (b + 1) * block)) for b in chosen]).astype(np.int32)


def ranges(sel: np.ndarray):
    """Maximal contiguous [start, end) ranges of an ascending index list."""
    sel = np.asarray(sel)
    if sel.size == 0:
        return []
    cut = np.nonzero(np.diff(sel) != 1)[0]
    starts = np.concatenate([[0], cut + 1])
    ends = np.concatenate([cut + 1, [sel.size]])
    return [(int(sel[a]), int(sel[b - 1]) + 1) for a, b in zip(starts, ends)]
