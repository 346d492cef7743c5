"""GPU parity of sffn_prefill (token-selective FFN) against the fp64 oracle:
unselected rows are Y = bf16(X + Y_attn) bit for bit; selected rows match
bf16(Y + FFN(Y)) within relative L2 1e-2 per row (H is rounded to bf16 as a
GEMM input, the oracle keeps fp64)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import ffn_from_layer, mat_from_act
from tests.parity import layer_to

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def sffn():
    from activation_sparse_ffn_gemv_gb300 import sffn as S
    S.lib()
    return S


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_prefill(sffn, layer_cpu, X, Ya, m, recent_n=128, min_keep=1):
    layer = layer_to(layer_cpu, "cuda")
    w = sffn.Weights(layer)
    Xd, Yad = X.cuda(), Ya.cuda()
    sel, n = sffn.token_select(Yad, m, recent_n, min_keep)
    out = sffn.prefill(Xd, Yad, w, sel, n)
    ws = sffn.alloc_workspace(sffn.WS_PREFILL, X.shape[0], w)
    out2 = sffn.prefill(Xd, Yad, w, sel, n, workspace=ws)
    torch.cuda.synchronize()
    assert sffn.read_device_error(ws) == 0
    assert torch.equal(out, out2), "prefill is not deterministic"
    k = int(n.item())
    return out.cpu(), sel[:k].cpu().numpy()


def check_prefill(sffn, layer_cpu, X, Ya, m, sample_selected=None, nthreads=16, recent_n=128, tol=None):
    L = X.shape[0]
    out, sel = run_prefill(sffn, layer_cpu, X, Ya, m, recent_n=recent_n)
    ob = _bits(out)
    Xm, Yam = mat_from_act(X), mat_from_act(Ya)
    Y = O.residual(Xm, Yam)
    mask = np.zeros(L, np.uint8)
    mask[sel] = 1
    # unselected rows: Z = 0, out = Y bit for bit
    uns = mask == 0
    assert np.array_equal(ob[uns], Y[uns])
    rows = sel if sample_selected is None else np.random.default_rng(0).choice(sel, min(sample_selected, sel.size),
                                                                                replace=False)
    rows = np.sort(rows).astype(np.int32)
    z, _ = O.prefill_rows(ffn_from_layer(layer_cpu), Xm, Yam, mask, rows, nthreads=nthreads)
    ref = Y[rows].astype(np.uint32) << 16
    ref = ref.view(np.float32).astype(np.float64) + z
    got = (ob[rows].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
    tol = TOL if tol is None else tol
    assert err.max() <= tol, f"max row relative L2 error {err.max():.3e}"
    return sel, err


SMALL = [
    # (L, d, F, m)
    (200, 256, 256, 0.5),
    (333, 320, 384, 0.3),
    (128, 128, 128, 1.0),
    (600, 512, 640, 0.7),
    (77, 192, 256, 0.0),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_prefill_small(sffn, case):
    L, d, F, m = case
    layer = W.make_ffn_layer(5, seed=3, d_model=d, d_ff=F)
    X, Ya = W.make_prefill_inputs(L, d, seed=L)
    sel, err = check_prefill(sffn, layer, X, Ya, m, recent_n=16)
    if m == 1.0:
        assert sel.size == L


def test_prefill_many_tiles(sffn):
    # several m-tiles and n-tiles with ragged edges in both
    L, d, F = 1500, 384, 1280
    layer = W.make_ffn_layer(5, seed=5, d_model=d, d_ff=F)
    X, Ya = W.make_prefill_inputs(L, d, seed=11)
    check_prefill(sffn, layer, X, Ya, 0.6, sample_selected=96, recent_n=40)


def test_prefill_single_selected_token(sffn):
    L, d, F = 300, 256, 256
    layer = W.make_ffn_layer(5, seed=6, d_model=d, d_ff=F)
    X, _ = W.make_prefill_inputs(L, d, seed=12)
    Ya = torch.zeros(L, d, dtype=torch.bfloat16)
    Ya[17, 3] = 5.0
    sel, _ = check_prefill(sffn, layer, X, Ya, 0.5, recent_n=0)
    assert sel.tolist() == [17]


@pytest.mark.slow
@pytest.mark.parametrize("m", [0.2, 1.0])
def test_config_prefill_full(sffn, m):
    c = W.CONFIGS[5]
    layer = W.make_ffn_layer(5, seed=0)
    X, Ya = W.make_prefill_inputs(c["L"], c["d_model"], seed=0)
    sel, err = check_prefill(sffn, layer, X, Ya, m, sample_selected=12, nthreads=16, recent_n=c["recent_n"])
    if m == 1.0:
        assert sel.size == c["L"]


# int4-g64 weights: the GEMMs' dequantising warps form code * scale rounded once
# to bf16 (relative 2^-9 per weight, as H's rounding), so the int4 bound of the
# decode, 2e-2, applies.
INT4 = [
    # (L, d, F, m)
    (300, 512, 512, 0.3),
    (200, 320, 384, 1.0),      # d_model 320: the down GEMM's last n-tile is partial
    (700, 256, 1280, 0.6),     # several m- and n-tiles
]


@pytest.mark.parametrize("case", INT4, ids=lambda c: "-".join(map(str, c)))
def test_int4_prefill(sffn, case):
    L, d, F, m = case
    layer = W.make_ffn_layer(4, seed=7, d_model=d, d_ff=F)
    assert layer["wdtype"] == "int4_g64" and layer.get("b_gate") is None
    X, Ya = W.make_prefill_inputs(L, d, seed=L + 1)
    sel, err = check_prefill(sffn, layer, X, Ya, m, recent_n=16, tol=2e-2)
    if m == 1.0:
        assert sel.size == L


def test_int4_prefill_workload_shape(sffn):
    # the int4 decode workload's layer (d_model 2048, d_ff 11008), 2048 tokens
    layer = W.make_ffn_layer(4, seed=8)
    X, Ya = W.make_prefill_inputs(2048, 2048, seed=8)
    check_prefill(sffn, layer, X, Ya, 0.5, sample_selected=12, recent_n=64, tol=2e-2)
