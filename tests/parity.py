"""Comparison helpers: CUDA path vs the fp64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from tests.oracle_io import ffn_from_layer, mat_from_act

TIE_REL = 1e-6   # selection: elements within 1e-6 (relative) of the cut are exempt
TOL = {"f32": 1e-5, "bf16": 1e-2, "int4_g64": 2e-2}   # per-token relative L2 bound on outputs

_MODE = {"exact": O.EXACT, "threshold": O.THRESHOLD, "keep_ratio": O.KEEP_RATIO}
_SCORE = {"gate": O.SCORE_GATE, "gate_up": O.SCORE_GATE_UP}


def layer_to(layer: dict, device) -> dict:
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in layer.items()}


def sets_from(active_idx: np.ndarray, n_active: np.ndarray):
    return [active_idx[b, : n_active[b]] for b in range(n_active.shape[0])]


def check_selection(gpu_sets, ref, mode: str, F: int, keep_k: int | None = None):
    """Bit-exact sets except for elements within the tie band of the cut.
    Returns the number of exempted elements."""
    exempt = 0
    for b, gs in enumerate(gpu_sets):
        assert gs.size == 0 or (np.all(np.diff(gs) > 0) and gs[0] >= 0 and gs[-1] < F), "not ascending / in range"
        rs = ref["active_idx"][b, : ref["n_active"][b]]
        diff = np.setxor1d(gs, rs)
        if diff.size:
            q = ref["g"][b] if mode == "exact" else ref["score"][b]
            cut = 0.0 if mode == "exact" else ref["cut"][b]
            band = TIE_REL * np.maximum(abs(cut), ref["cond"][b][diff])
            bad = diff[np.abs(q[diff] - cut) > band]
            assert bad.size == 0, (f"token {b}: {bad.size} set differences outside the tie band, e.g. "
                                   f"j={bad[:5].tolist()} q={q[bad[:5]].tolist()} cut={cut}")
            exempt += diff.size
        if keep_k is not None:
            assert gs.size == keep_k, (gs.size, keep_k)
    return exempt


def check_outputs(gpu_out: np.ndarray, ref_out: np.ndarray, tol: float):
    """Per-token relative L2 error <= tol; an all-zero reference needs an all-zero output."""
    errs = []
    for b in range(ref_out.shape[0]):
        rn = np.linalg.norm(ref_out[b])
        if rn == 0.0:
            assert not np.any(gpu_out[b]), f"token {b}: reference is 0 but output is not"
            errs.append(0.0)
            continue
        errs.append(np.linalg.norm(gpu_out[b] - ref_out[b]) / rn)
    assert max(errs) <= tol, f"max relative L2 error {max(errs):.3e} > {tol:.1e}"
    return max(errs)


def run_and_check_decode(sffn, layer_cpu: dict, x_cpu: torch.Tensor, mode: str, score: str = "gate",
                         param: float = 0.0, nthreads: int = 8, out_tol: float | None = None,
                         batch: int = 8, max_exempt: int | None = None):
    """Runs sffn_decode on the GPU (``batch`` tokens per call) and checks sets +
    outputs against the oracle.  At most ``max_exempt`` set elements (default:
    two per token) may differ inside the tie band: the band only forgives
    rounding at the cut, so a systematic error near the cut still fails."""
    dev = "cuda"
    layer = layer_to(layer_cpu, dev)
    w = sffn.Weights(layer)
    if mode != "exact":
        w.set_down_norms(sffn.down_norms(w))
    x = x_cpu.to(dev)
    outs, idxs, ns = [], [], []
    for t0 in range(0, x.shape[0], batch):
        o, i, nn = sffn.decode(x[t0:t0 + batch], w, {"exact": 0, "threshold": 1, "keep_ratio": 2}[mode],
                               {"gate": 0, "gate_up": 1}[score], param)
        outs.append(o)
        idxs.append(i)
        ns.append(nn)
    out, idx, n = torch.cat(outs), torch.cat(idxs), torch.cat(ns)
    torch.cuda.synchronize()
    idx, n = idx.cpu().numpy(), n.cpu().numpy()
    gpu_sets = sets_from(idx, n)
    ffn, xm = ffn_from_layer(layer_cpu), mat_from_act(x_cpu)
    B, F = x_cpu.shape[0], layer_cpu["d_ff"]
    gi = np.zeros((B, F), np.int32)
    for b, s in enumerate(gpu_sets):
        gi[b, : s.size] = s
    ref = O.decode(ffn, xm, _MODE[mode], _SCORE[score], param, given_idx=gi, given_n=n.astype(np.int32),
                   nthreads=nthreads, details=True)
    keep_k = O.keep_count(F, param) if mode == "keep_ratio" else None
    exempt = check_selection(gpu_sets, ref, mode, F, keep_k)
    limit = 2 * B if max_exempt is None else max_exempt
    assert exempt <= limit, f"{exempt} set elements differ inside the tie band (limit {limit})"
    err = check_outputs(out.float().cpu().numpy().astype(np.float64), ref["out"],
                        out_tol if out_tol is not None else TOL[layer_cpu["wdtype"]])
    return dict(exempt=exempt, err=err, n_active=n, ref=ref, out=out)
