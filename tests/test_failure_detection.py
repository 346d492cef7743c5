"""Failure detection without a GPU fault: every device-side wait is bounded and
every index the device receives is range-checked, and both outcomes land in the
workspace's error word, which sffn_read_device_error returns (and clears).

* The decode call's CTAs meet at a grid barrier whose wait gives up after about
  one second.  Setting the barrier's base one arrival beyond what the call can
  reach (a value no call writes) makes the wait run out: the call records
  SFFN_ERR_TIMEOUT, its CTAs return, and after the error is read (which resets
  the barrier counters) the next call is correct again.
* Prefill receives the selection from the caller: a count above L is clamped
  and an out-of-range token index is skipped, each recorded as SFFN_ERR_DEVICE,
  while every other row is computed as usual.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.parity import layer_to

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def S():
    from activation_sparse_ffn_gemv_gb300 import build as B
    B.build()
    from activation_sparse_ffn_gemv_gb300 import sffn
    sffn.lib()
    return sffn


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


# (config, weights): bf16 runs the streaming gate kernel; int4 with one token runs
# the staged single-token kernel, and its dense layer the int4 stream kernel
TIMEOUT_CASES = {"bf16": (2, "exact"), "int4": (4, "exact"), "int4_dense": (4, "dense")}


@pytest.mark.parametrize("case", list(TIMEOUT_CASES))
def test_decode_barrier_timeout_is_reported_and_recovers(S, case):
    cfg, kind = TIMEOUT_CASES[case]
    layer = layer_to(W.make_ffn_layer(cfg, seed=51, d_model=512, d_ff=2048), "cuda")
    w = S.Weights(layer)
    x = W.make_tokens(cfg, 1, seed=51, d_model=512).cuda()
    ws = S.alloc_workspace(S.WS_DECODE, 1, w)
    ctl = ws[:16].view(torch.int32)   # error word, barrier arrivals, arrivals before the call

    def call():
        if kind == "dense":
            return S.decode_dense(x, w, workspace=ws), None, None
        return S.decode(x, w, S.MODE_EXACT, workspace=ws)

    ref, ref_idx, ref_n = call()
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == 0
    ref, ref_idx, ref_n = call()
    torch.cuda.synchronize()
    arrivals = int(ctl[1].item())
    assert arrivals > 0 and int(ctl[2].item()) == arrivals  # the pair a finished call leaves
    # a base one past the arrivals: this call's CTAs can never all be counted
    ctl[2] = arrivals + 1
    torch.cuda.synchronize()
    call()
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == S.ERR_TIMEOUT
    assert int(ctl.abs().sum().item()) == 0  # reading the error reset the control block
    out, idx, n = call()
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == 0
    if n is not None:
        assert torch.equal(n, ref_n) and torch.equal(idx[0, : int(n[0])], ref_idx[0, : int(n[0])])
    assert np.array_equal(_bits(out), _bits(ref))


def _prefill_setup(S, L=300, d=256, F=512):
    layer = layer_to(W.make_ffn_layer(5, seed=61, d_model=d, d_ff=F), "cuda")
    w = S.Weights(layer)
    X, Ya = W.make_prefill_inputs(L, d, seed=61)
    return w, X.cuda(), Ya.cuda()


def test_prefill_count_above_length_is_clamped_and_reported(S):
    w, X, Ya = _prefill_setup(S)
    L = X.shape[0]
    sel = torch.arange(L, dtype=torch.int32, device="cuda")
    ws = S.alloc_workspace(S.WS_PREFILL, L, w)
    ref = S.prefill(X, Ya, w, sel, torch.tensor([L], dtype=torch.int32, device="cuda"), workspace=ws)
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == 0
    out = S.prefill(X, Ya, w, sel, torch.tensor([L + 5], dtype=torch.int32, device="cuda"), workspace=ws)
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == S.ERR_DEVICE
    assert np.array_equal(_bits(out), _bits(ref))   # clamped to every token


def test_prefill_out_of_range_index_is_skipped_and_reported(S):
    w, X, Ya = _prefill_setup(S)
    L = X.shape[0]
    ws = S.alloc_workspace(S.WS_PREFILL, L, w)
    good = torch.tensor([0, 5, 10, 299], dtype=torch.int32, device="cuda")
    ref = S.prefill(X, Ya, w, good, torch.tensor([4], dtype=torch.int32, device="cuda"), workspace=ws)
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == 0
    bad = torch.tensor([0, 5, L + 3, 10, 299], dtype=torch.int32, device="cuda")
    out = S.prefill(X, Ya, w, bad, torch.tensor([5], dtype=torch.int32, device="cuda"), workspace=ws)
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == S.ERR_DEVICE
    ob, rb = _bits(out), _bits(ref)
    # the valid selected rows get their FFN, every other row is the residual;
    # the rows' values do not depend on which other rows share their tile
    assert np.array_equal(ob, rb)
    # and the other rows are the residual (an empty selection gives it for all)
    Y = _bits(S.prefill(X, Ya, w, good, torch.tensor([0], dtype=torch.int32, device="cuda"), workspace=ws))
    torch.cuda.synchronize()
    assert S.read_device_error(ws) == 0
    rest = np.setdiff1d(np.arange(L), [0, 5, 10, 299])
    assert np.array_equal(ob[rest], Y[rest])
    assert not np.array_equal(ob[[0, 5, 10, 299]], Y[[0, 5, 10, 299]])
