"""Low-rank gate predictor -- TEST INFRASTRUCTURE (the fp64 oracle's part for it).

Only the tests may import this module; the product path never does.

The denseflux write-up ("denseflux: skipping most of a dense FFN", the gate
predictor discussion) notes that exact gating must read all of W_gate, a third of
the FFN bytes, and that a predictor may skip even that; its best untrained
predictor is low-rank.  Read plainly:

  * offline: W_gate ~= A B with A = U_r diag(S_r) [F, r] and B = V_r^T [r, d],
    the rank-r truncated SVD of the (dequantised) gate matrix;
  * per token: predicted pre-activation p = A (B x) + b;
  * candidates P(alpha) = { j : p_j >= -alpha } (alpha >= 0 widens the set:
    recall for bytes; alpha = +inf keeps every neuron);
  * the exact gate is formed only for j in P; a candidate is active under the
    layer's exact rule (act(g_j) != 0); a neuron outside P is skipped even if it
    would have been active (a miss);
  * out = sum over the active candidates of act(g_j) u_j W_down[:, j].

Bytes read per token: the fp32 factors 4 r (F + d), and, in the weights'
storage element size, the candidates' gate rows |P| d and the active W_up rows
and W_down columns 2 |active| d (bias, x and out come on top, as in the exact
decode).

Pinned by tests/test_predictor_oracle.py: alpha = +inf reduces to the exact
decode; a gate matrix of exact rank r is predicted with full recall by rank r;
full-rank factors reproduce the gate; candidate sets grow with alpha; no
candidate gives a zero output.
"""
from __future__ import annotations

import numpy as np

from . import EXACT, FFN, INT4_G64, Mat, decode


def lowrank_factors(w_gate: np.ndarray, r: int):
    """Rank-r factors (A [F, r], B [r, d]) of w_gate [F, d] (fp64) by truncated SVD."""
    w = np.asarray(w_gate, np.float64)
    U, S, Vt = np.linalg.svd(w, full_matrices=False)
    r = int(max(0, min(r, S.size)))
    return U[:, :r] * S[:r], Vt[:r].copy()


def predict(A: np.ndarray, B: np.ndarray, bias, x: np.ndarray) -> np.ndarray:
    """Predicted gate pre-activations p [T, F] for tokens x [T, d] (fp64)."""
    x = np.atleast_2d(np.asarray(x, np.float64))
    p = (x @ B.T) @ A.T
    if bias is not None:
        p = p + np.asarray(bias, np.float64)[None, :]
    return p


def candidates(p_row: np.ndarray, alpha: float) -> np.ndarray:
    """Ascending indices j with p_j >= -alpha."""
    if alpha == np.inf:
        return np.arange(p_row.size, dtype=np.int32)
    return np.nonzero(p_row >= -alpha)[0].astype(np.int32)


def decode_predicted(ffn: FFN, x: Mat, A: np.ndarray, B: np.ndarray, alpha: float, nthreads: int = 1):
    """Exact gating restricted to the predicted candidates.  Returns a dict with
    ``out`` [T, d] fp64, per-token ``candidates`` and ``active`` (ascending
    arrays), ``recall`` [T] (share of the exact rule's active neurons that are
    candidates; 1 when there are none) and ``bytes`` [T] for the element size of
    the stored weights."""
    T, F, d = x.rows, ffn.d_ff, ffn.d_model
    ref = decode(ffn, x, EXACT, details=True, nthreads=nthreads)
    bias = None if ffn.b_gate is None else np.asarray(ffn.b_gate, np.float64)
    p = predict(A, B, bias, x.to_f64())
    cands, acts, recall = [], [], np.ones(T)
    gi = np.zeros((T, F), np.int32)
    gn = np.zeros(T, np.int32)
    for t in range(T):
        c = candidates(p[t], alpha)
        act = c[ref["a"][t, c] != 0.0]
        cands.append(c)
        acts.append(act)
        gi[t, : act.size] = act
        gn[t] = act.size
        exact = ref["active_idx"][t, : ref["n_active"][t]]
        if exact.size:
            recall[t] = np.intersect1d(exact, c).size / exact.size
    out = decode(ffn, x, EXACT, given_idx=gi, given_n=gn, nthreads=nthreads)["out"] if T else np.zeros((0, d))
    esz = ffn.w_gate.data.dtype.itemsize if ffn.w_gate.fmt != INT4_G64 else 0.5 + 2.0 / 64
    r = A.shape[1]
    nbytes = np.array([esz * (c.size * d + 2 * a.size * d) + 4.0 * r * (F + d) for c, a in zip(cands, acts)])
    return {"out": out, "candidates": cands, "active": acts, "recall": recall, "bytes": nbytes, "p": p,
            "exact": ref}
