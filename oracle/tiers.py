"""Keep-ratio tier tables with a per-layer core set -- TEST INFRASTRUCTURE (the
fp64 oracle's part for them).  Only the tests may import this module.

The WiSparse write-up (kwkr.cn/news/623085, sec. 2.2, the paragraph after the
score definition) keeps k = F / M columns per token for tier M and suggests, to
switch less online, counting over a calibration set how often each column of a
layer is kept at a tier, taking the most frequent columns as a guaranteed base
("core") set, and completing each token's selection dynamically.  Read plainly:

  * offline: for tier k and core size c (0 <= c <= k), the core set is the c
    columns kept most often by the per-token top-k over the calibration tokens
    (count ties to the lower index); it is stored ascending;
  * online, per token: keep = core  U  the (k - c) largest scores among the
    columns outside the core (score ties to the lower index); ascending.

With c = 0 this is the plain keep-ratio selection; the online work is a top-
(k - c) over F - c candidates instead of a top-k over F.

Pinned by tests/test_tiers_oracle.py: c = 0 equals the keep-ratio selection of
the exact oracle; c = k returns the core; brute force over all subsets of size k
containing the core on small F; frequency counting on constructed calibrations.
"""
from __future__ import annotations

import numpy as np


def topk_lower_index(scores: np.ndarray, k: int, exclude=None) -> np.ndarray:
    """Indices of the k largest scores (ties to the lower index), ascending;
    columns in `exclude` are not candidates."""
    s = np.asarray(scores, np.float64)
    F = s.size
    cand = np.ones(F, bool)
    if exclude is not None and len(exclude):
        cand[np.asarray(exclude, np.int64)] = False
    idx = np.nonzero(cand)[0]
    k = int(max(0, min(k, idx.size)))
    if k == 0:
        return np.zeros(0, np.int32)
    # order by (score descending, index ascending)
    order = np.lexsort((idx, -s[idx]))
    return np.sort(idx[order[:k]]).astype(np.int32)


def core_set(calib_scores: np.ndarray, k: int, c: int) -> np.ndarray:
    """The c columns most often in a calibration token's top-k (ties lower index), ascending."""
    S = np.atleast_2d(np.asarray(calib_scores, np.float64))
    N, F = S.shape
    freq = np.zeros(F, np.int64)
    for t in range(N):
        freq[topk_lower_index(S[t], k)] += 1
    c = int(max(0, min(c, F)))
    order = np.lexsort((np.arange(F), -freq))
    return np.sort(order[:c]).astype(np.int32)


def select_with_core(scores: np.ndarray, k: int, core: np.ndarray) -> np.ndarray:
    """core U the (k - |core|) largest scores outside the core, ascending."""
    core = np.asarray(core, np.int32)
    extra = topk_lower_index(scores, k - core.size, exclude=core)
    return np.sort(np.concatenate([core, extra])).astype(np.int32)
