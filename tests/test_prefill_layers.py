"""GPU: a stack of token-selective prefill layers driven by the per-layer
schedule equals the same layers run one call at a time (bit for bit, selections
included); the dense tier keeps every token."""
from __future__ import annotations

import pytest
import torch

from activation_sparse_ffn_gemv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sffn():
    from activation_sparse_ffn_gemv_gb300 import sffn as S
    S.lib()
    return S


def _stack(sffn, n, L=300, d=256, F=256):
    layers = [{k: (v.cuda() if torch.is_tensor(v) else v) for k, v in
               W.make_ffn_layer(5, seed=50 + i, d_model=d, d_ff=F).items()} for i in range(n)]
    ws = [sffn.Weights(l) for l in layers]
    X, _ = W.make_prefill_inputs(L, d, seed=1)
    yas = [W.make_prefill_inputs(L, d, seed=10 + i)[1].cuda() for i in range(n)]
    return layers, ws, X.cuda(), yas


@pytest.mark.parametrize("n,first", [(3, 0), (4, 0), (2, 2)])
def test_stack_equals_chained_layers(sffn, n, first):
    layers, ws, x0, yas = _stack(sffn, n)
    L = x0.shape[0]
    s = sffn.schedule(dense_until=1, mass_thresh=0.5, recent_n=16, deep_layer_start=3, mass_thresh_deep=0.2)
    wsp = torch.zeros(max(int(sffn.lib().sffn_prefill_layers_workspace_size(L, w.ref())) for w in ws),
                      dtype=torch.uint8, device="cuda")
    out, sel, ns = sffn.prefill_layers(x0, yas, ws, s, first_layer=first, workspace=wsp)
    x = x0
    for i in range(n):
        m = sffn.schedule_mass(s, first + i)
        si, ni = sffn.token_select(yas[i], m, s.recent_n, s.min_keep)
        x = sffn.prefill(x, yas[i], ws[i], si, ni)
        torch.cuda.synchronize()
        k = int(ni.item())
        assert int(ns[i].item()) == k, f"layer {first + i}: n_sel"
        assert torch.equal(sel[i, :k], si[:k]), f"layer {first + i}: selection"
        if first + i < s.dense_until:
            assert k == L  # the dense tier keeps every token
    torch.cuda.synchronize()
    assert torch.equal(out, x)
    assert sffn.read_device_error(wsp) == 0
    # deep layers keep fewer tokens than middle ones at the same inputs' scale
    masses = [sffn.schedule_mass(s, first + i) for i in range(n)]
    if 0.2 in [round(m, 3) for m in masses] and 0.5 in [round(m, 3) for m in masses]:
        nd = [int(ns[i]) for i in range(n) if round(masses[i], 3) == 0.2]
        nm = [int(ns[i]) for i in range(n) if round(masses[i], 3) == 0.5]
        assert max(nd) < L and min(nm) < L


def test_dense_preset_equals_dense_ffn(sffn):
    # every layer dense: the stack's output is the chained full-token prefill
    layers, ws, x0, yas = _stack(sffn, 2)
    L = x0.shape[0]
    out, sel, ns = sffn.prefill_layers(x0, yas, ws, sffn.schedule_preset("dense"))
    all_idx = torch.arange(L, dtype=torch.int32, device="cuda")
    x = x0
    for i in range(2):
        x = sffn.prefill(x, yas[i], ws[i], all_idx, torch.tensor([L], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert (ns == L).all()
    assert torch.equal(out, x)


def _oracle_stack(layers_cpu, X, yas_cpu, sels):
    """The oracle's layers chained on the GPU's selections: each layer's
    output rows are bf16(Y + FFN(Y)) for the selected tokens and Y = bf16(X +
    Y_attn) for the rest, and feed the next layer as its X."""
    import numpy as np

    import oracle as O
    from tests.oracle_io import ffn_from_layer, mat_from_act
    x = X
    for i, layer in enumerate(layers_cpu):
        Xm, Yam = mat_from_act(x), mat_from_act(yas_cpu[i])
        Y = O.residual(Xm, Yam)
        mask = np.zeros(x.shape[0], np.uint8)
        mask[sels[i]] = 1
        nxt = Y.copy()
        if sels[i].size:
            _, ob = O.prefill_rows(ffn_from_layer(layer), Xm, Yam, mask, sels[i], nthreads=8)
            nxt[sels[i]] = ob
        x = torch.from_numpy(nxt.view(np.int16)).view(torch.bfloat16)
    return x


@pytest.mark.parametrize("n,first", [(3, 0), (4, 1)])
def test_stack_matches_the_oracle_chained(sffn, n, first):
    # each layer's selection against the oracle's mass rule (tie band as the
    # selection tests), then the stack's output against the oracle's layers
    # chained on those selections: relative L2 per row within 1e-2 per layer
    import numpy as np

    import oracle as O
    from tests.oracle_io import mat_from_act
    from tests.test_select_parity import check_select
    L, d, F = 300, 256, 256
    layers_cpu = [W.make_ffn_layer(5, seed=70 + i, d_model=d, d_ff=F) for i in range(n)]
    ws = [sffn.Weights({k: (v.cuda() if torch.is_tensor(v) else v) for k, v in l.items()}) for l in layers_cpu]
    X, _ = W.make_prefill_inputs(L, d, seed=2)
    yas = [W.make_prefill_inputs(L, d, seed=20 + i)[1] for i in range(n)]
    s = sffn.schedule(dense_until=1, mass_thresh=0.5, recent_n=16, deep_layer_start=3, mass_thresh_deep=0.2)
    out, sel, ns = sffn.prefill_layers(X.cuda(), [y.cuda() for y in yas], ws, s, first_layer=first)
    torch.cuda.synchronize()
    sels = []
    for i in range(n):
        k = int(ns[i].item())
        gs = sel[i, :k].cpu().numpy()
        m = sffn.schedule_mass(s, first + i)
        want, _, _ = check_select(sffn, yas[i], m, s.recent_n, s.min_keep)
        assert np.array_equal(gs, want), f"layer {first + i}: the stack's selection differs from the single call"
        sels.append(gs)
    ref = _oracle_stack(layers_cpu, X, yas, sels)
    got = out.cpu().float().numpy().astype(np.float64)
    want = ref.float().numpy().astype(np.float64)
    err = np.linalg.norm(got - want, axis=1) / np.maximum(np.linalg.norm(want, axis=1), 1e-30)
    assert err.max() <= 1e-2 * n, f"max row relative L2 error {err.max():.3e} after {n} layers"
