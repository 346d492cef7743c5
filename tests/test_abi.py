"""The C-ABI boundary: the library loads and exports every symbol the header
declares (CPU), host-side argument checks return the documented status before
anything is launched (CPU where no CUDA call is reached, GPU otherwise)."""
from __future__ import annotations

import ctypes as C
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sffn.h")


@pytest.fixture(scope="module")
def S():
    from activation_sparse_ffn_gemv_gb300 import build as B
    B.build()
    from activation_sparse_ffn_gemv_gb300 import sffn
    sffn.lib()
    return sffn


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sffn_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ("sffn_decode", "sffn_token_select", "sffn_prefill", "sffn_workspace_size",
                 "sffn_status_string", "sffn_down_norms", "sffn_read_device_error"):
        assert must in names


def test_library_exports_every_declared_symbol(S):
    lib = C.CDLL(S.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(S):
    for st in range(9):
        assert S.status_string(st) and S.status_string(st) != "unknown status"
    assert S.status_string(99) == "unknown status"


def test_null_arguments_rejected_before_any_cuda_call(S):
    L = S.lib()
    w = S.FFNWeights(S.BF16, S.ACT_RELU, 64, 128, 16, 16, 16, None, None, None, None, None)
    # x == NULL
    assert L.sffn_decode(None, 1, C.byref(w), 0, 0, 0.0, 16, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    # unknown mode / score
    assert L.sffn_decode(16, 1, C.byref(w), 7, 0, 0.0, 16, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    assert L.sffn_decode(16, 1, C.byref(w), 0, 5, 0.0, 16, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    # weights struct missing
    assert L.sffn_decode(16, 1, None, 0, 0, 0.0, 16, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    # token select / prefill null pointers
    assert L.sffn_token_select(None, 16, 64, 0.5, 4, 1, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    assert L.sffn_prefill(None, 16, 16, C.byref(w), 16, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    assert L.sffn_down_norms(None, 16, None) == S.ERR_INVALID_ARG


def test_shape_and_parameter_checks_before_any_cuda_call(S):
    L = S.lib()

    def wts(**kw):
        f = dict(wdtype=S.BF16, act=S.ACT_RELU, d_model=64, d_ff=128)
        f.update(kw)
        return S.FFNWeights(f["wdtype"], f["act"], f["d_model"], f["d_ff"], 16, 16, 16, 16, 16, 16, None, 16)

    def dec(w, B=1, mode=0, param=0.0, x=16):
        return L.sffn_decode(x, B, C.byref(w), mode, 0, param, 16, 16, 16, 256, 1 << 20, None)

    assert dec(wts(d_model=12)) == S.ERR_SHAPE                 # d % 8
    assert dec(wts(d_model=96, wdtype=S.INT4_G64)) == S.ERR_SHAPE  # int4 needs d % 64
    assert dec(wts(d_ff=0)) == S.ERR_SHAPE
    assert dec(wts(), B=0) == S.ERR_SHAPE
    assert dec(wts(), B=9) == S.ERR_SHAPE
    assert dec(wts(d_model=8192)) == S.ERR_SHAPE               # decode limit 4096
    assert dec(wts(), x=8) == S.ERR_ALIGNMENT
    assert dec(wts(), mode=2, param=0.0) == S.ERR_INVALID_ARG  # keep ratio in (0, 1]
    assert dec(wts(), mode=2, param=1.5) == S.ERR_INVALID_ARG
    assert dec(wts(), mode=1, param=-1.0) == S.ERR_INVALID_ARG # tau >= 0
    assert dec(wts(act=5)) == S.ERR_INVALID_ARG
    assert L.sffn_token_select(16, 0, 64, 0.5, 4, 1, 16, 16, 256, 1 << 20, None) == S.ERR_SHAPE
    assert L.sffn_token_select(16, 16, 64, 0.5, -1, 1, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    assert L.sffn_token_select(16, 16, 64, 0.5, 4, 0, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    assert L.sffn_token_select(8, 16, 64, 0.5, 4, 1, 16, 16, 256, 1 << 20, None) == S.ERR_ALIGNMENT
    w = wts(act=S.ACT_SILU)
    assert L.sffn_prefill(16, 16, 16, C.byref(wts()), 16, 16, 16, 256, 1 << 20, None) == S.ERR_UNSUPPORTED  # ReLU
    assert L.sffn_prefill(16, 16, 0, C.byref(w), 16, 16, 16, 256, 1 << 20, None) == S.ERR_SHAPE
    assert L.sffn_workspace_size(5, 1, None) == 0


def test_noalloc_reports_argument_errors_like_decode(S):
    # sffn_decode_noalloc runs sffn_decode's own checks, in the same order, before
    # it touches its built-in array: every bad argument gives the same status
    L = S.lib()

    def wts(**kw):
        f = dict(wdtype=S.BF16, act=S.ACT_RELU, d_model=64, d_ff=128)
        f.update(kw)
        return S.FFNWeights(f["wdtype"], f["act"], f["d_model"], f["d_ff"], 16, 16, 16, 16, 16, 16, None, 16)

    cases = [  # (weights, B, mode, score, param, x, out)
        (wts(d_model=12), 1, 0, 0, 0.0, 16, 16), (wts(d_model=96, wdtype=S.INT4_G64), 1, 0, 0, 0.0, 16, 16),
        (wts(d_ff=0), 1, 0, 0, 0.0, 16, 16), (wts(d_ff=70000), 1, 0, 0, 0.0, 16, 16),
        (wts(), 0, 0, 0, 0.0, 16, 16), (wts(), 9, 0, 0, 0.0, 16, 16), (wts(d_model=8192), 1, 0, 0, 0.0, 16, 16),
        (wts(), 1, 0, 0, 0.0, 8, 16), (wts(), 1, 0, 0, 0.0, 16, 8), (wts(), 1, 2, 0, 0.0, 16, 16),
        (wts(), 1, 2, 0, 1.5, 16, 16), (wts(), 1, 1, 0, -1.0, 16, 16), (wts(act=5), 1, 0, 0, 0.0, 16, 16),
        (wts(), 1, 7, 0, 0.0, 16, 16), (wts(), 1, 0, 5, 0.0, 16, 16), (wts(), 1, 0, 0, 0.0, None, 16),
        (wts(), 1, 0, 0, 0.0, 16, None), (wts(wdtype=S.INT4_G64, d_model=512), 1, 2, 0, 0.5, 16, 16),
        (wts(wdtype=S.INT4_G64, d_model=576), 1, 0, 0, 0.0, 16, 16),
    ]
    for w, B, mode, score, param, x, out in cases:
        a = L.sffn_decode(x, B, C.byref(w), mode, score, param, out, 16, 16, 256, 1 << 20, None)
        b = L.sffn_decode_noalloc(x, B, C.byref(w), mode, score, param, out, 16, 16, None)
        assert a == b and a != S.OK, (a, b)
    assert L.sffn_decode_noalloc(16, 1, None, 0, 0, 0.0, 16, 16, 16, None) == S.ERR_INVALID_ARG
    assert L.sffn_decode_noalloc_read_error(None, None) == S.ERR_INVALID_ARG


def test_gate_scores_argument_checks(S):
    # sffn_gate_scores takes the decode's checks for the threshold rule (down
    # norms required) and its own scores pointer, all before any CUDA call
    L = S.lib()

    def wts(norms=16, **kw):
        f = dict(wdtype=S.BF16, act=S.ACT_SILU, d_model=512, d_ff=128)
        f.update(kw)
        return S.FFNWeights(f["wdtype"], f["act"], f["d_model"], f["d_ff"], 16, 16, 16, 16, 16, 16, None, norms)

    def gs(w, B=1, score=0, x=16, scores=16):
        return L.sffn_gate_scores(x, B, C.byref(w), score, scores, 256, 1 << 20, None)

    assert gs(wts(), x=None) == S.ERR_INVALID_ARG
    assert gs(wts(), scores=None) == S.ERR_INVALID_ARG
    assert gs(wts(), score=5) == S.ERR_INVALID_ARG
    assert gs(wts(norms=None)) == S.ERR_INVALID_ARG   # the score needs ||W_down[:, j]||
    assert gs(wts(norms=8)) == S.ERR_ALIGNMENT
    assert gs(wts(), B=0) == S.ERR_SHAPE
    assert gs(wts(), B=9) == S.ERR_SHAPE
    assert gs(wts(d_model=8192)) == S.ERR_SHAPE
    assert gs(wts(wdtype=S.INT4_G64, d_model=576)) == S.ERR_SHAPE  # int4 rows: d % 512
    assert gs(wts(), x=8) == S.ERR_ALIGNMENT
    assert L.sffn_gate_scores(16, 1, None, 0, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG


def test_dense_layer_argument_checks(S):
    L = S.lib()

    def wts(**kw):
        f = dict(wdtype=S.BF16, act=S.ACT_RELU, d_model=512, d_ff=128)
        f.update(kw)
        return S.FFNWeights(f["wdtype"], f["act"], f["d_model"], f["d_ff"], 16, 16, 16, 16, 16, 16, None, None)

    def dense(w, B=1, x=16, out=16):
        return L.sffn_decode_dense(x, B, C.byref(w), out, 256, 1 << 20, None)

    assert dense(wts(), x=None) == S.ERR_INVALID_ARG
    assert dense(wts(), out=None) == S.ERR_INVALID_ARG
    assert dense(wts(), out=8) == S.ERR_ALIGNMENT
    assert dense(wts(), B=9) == S.ERR_SHAPE
    assert dense(wts(wdtype=S.F32)) == S.ERR_UNSUPPORTED
    assert dense(wts(d_model=8192)) == S.ERR_SHAPE
    assert L.sffn_decode_dense(16, 1, None, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG


def test_predicted_decode_argument_checks(S):
    # every check before the device is touched (on a machine without a GPU a
    # call that passes them all stops at the device check: ERR_CUDA)
    L = S.lib()
    inf = float("inf")

    def wts(**kw):
        f = dict(wdtype=S.BF16, act=S.ACT_RELU, d_model=64, d_ff=128)
        f.update(kw)
        return S.FFNWeights(f["wdtype"], f["act"], f["d_model"], f["d_ff"], 16, 16, 16, 16, 16, 16, None, None)

    def pred(w, x=16, fa=16, fb=16, rank=8, alpha=0.5, out=16, idx=16, n=16):
        return L.sffn_decode_predicted(x, C.byref(w), fa, fb, rank, alpha, out, idx, n, 256, 1 << 20, None)

    assert pred(wts(), x=None) == S.ERR_INVALID_ARG
    assert pred(wts(), out=None) == S.ERR_INVALID_ARG
    assert pred(wts(), idx=None) == S.ERR_INVALID_ARG
    assert pred(wts(), n=None) == S.ERR_INVALID_ARG
    assert pred(wts(), out=8) == S.ERR_ALIGNMENT
    assert pred(wts(wdtype=S.INT4_G64, d_model=512)) == S.ERR_UNSUPPORTED
    assert pred(wts(), alpha=-0.5) == S.ERR_INVALID_ARG
    assert pred(wts(), alpha=float("nan")) == S.ERR_INVALID_ARG
    assert pred(wts(), fa=None) == S.ERR_INVALID_ARG
    assert pred(wts(), fb=None) == S.ERR_INVALID_ARG
    assert pred(wts(), rank=0) == S.ERR_SHAPE
    assert pred(wts(), rank=129) == S.ERR_SHAPE          # rank <= d_ff
    assert pred(wts(), fb=24) == S.ERR_ALIGNMENT
    assert pred(wts(d_model=8192)) == S.ERR_SHAPE
    assert L.sffn_decode_predicted(16, None, 16, 16, 8, 0.5, 16, 16, 16, 256, 1 << 20, None) == S.ERR_INVALID_ARG
    # alpha = +inf: the factors are not read and may be null
    assert pred(wts(), fa=None, fb=None, rank=0, alpha=inf) not in (S.ERR_INVALID_ARG, S.ERR_SHAPE)


def test_tier_entry_points_argument_checks(S):
    L = S.lib()

    def wts(**kw):
        f = dict(wdtype=S.BF16, act=S.ACT_SILU, d_model=64, d_ff=128)
        f.update(kw)
        return S.FFNWeights(f["wdtype"], f["act"], f["d_model"], f["d_ff"], 16, 16, 16, 16, 16, 16, None, 16)

    def tiered(w, B=1, score=0, ratio=0.25, core=16, nc=4, x=16, out=16):
        return L.sffn_decode_tiered(x, B, C.byref(w), score, ratio, core, nc, out, 16, 16, 256, 1 << 20, None)

    assert tiered(wts(), x=None) == S.ERR_INVALID_ARG
    assert tiered(wts(), ratio=0.0) == S.ERR_INVALID_ARG
    assert tiered(wts(), ratio=1.5) == S.ERR_INVALID_ARG
    assert tiered(wts(), B=9) == S.ERR_SHAPE
    assert tiered(wts(wdtype=S.INT4_G64, d_model=576)) == S.ERR_SHAPE   # int4 rows: d_model % 512
    # the core is checked after the call's own arguments (on a machine without
    # a GPU those end at the device check)
    assert tiered(wts(), nc=-1) in (S.ERR_SHAPE, S.ERR_CUDA)
    assert tiered(wts(), core=None) in (S.ERR_INVALID_ARG, S.ERR_CUDA)

    def core_set(scores=16, N=4, F=128, k=16, c=8, core=16):
        return L.sffn_tier_core_set(scores, N, F, k, c, core, 256, 1 << 20, None)

    assert core_set(scores=None) == S.ERR_INVALID_ARG
    assert core_set(core=None) == S.ERR_INVALID_ARG
    assert core_set(N=0) == S.ERR_SHAPE
    assert core_set(F=70000) == S.ERR_SHAPE
    assert core_set(k=0) == S.ERR_INVALID_ARG
    assert core_set(k=129) == S.ERR_INVALID_ARG
    assert core_set(c=-1) == S.ERR_INVALID_ARG
    assert core_set(c=129) == S.ERR_INVALID_ARG
    assert L.sffn_tier_core_workspace_size(0, 128) == 0
    assert L.sffn_tier_core_workspace_size(4, 0) == 0
    assert L.sffn_tier_core_workspace_size(4, 128) > 0


@pytest.mark.gpu
def test_workspace_checks_on_gpu(S):
    from activation_sparse_ffn_gemv_gb300 import workloads as W
    layer = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in
             W.make_ffn_layer(2, seed=1, d_model=64, d_ff=128).items()}
    w = S.Weights(layer)
    x = W.make_tokens(2, 1, d_model=64).cuda()
    need = S.workspace_size(S.WS_DECODE, 1, w)
    assert need > 0
    ws = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(x)
    idx = torch.empty((1, 128), dtype=torch.int32, device="cuda")
    n = torch.empty(1, dtype=torch.int32, device="cuda")
    L = S.lib()
    st = L.sffn_decode(x.data_ptr(), 1, w.ref(), 0, 0, 0.0, out.data_ptr(), idx.data_ptr(), n.data_ptr(),
                       ws.data_ptr(), need - 1, None)
    assert st == S.ERR_WORKSPACE
    st = L.sffn_decode(x.data_ptr(), 1, w.ref(), 0, 0, 0.0, out.data_ptr(), idx.data_ptr(), n.data_ptr(),
                       ws.data_ptr() + 16, need, None)
    assert st == S.ERR_WORKSPACE           # not 256-byte aligned
    # threshold mode without down_norms
    st = L.sffn_decode(x.data_ptr(), 1, w.ref(), 1, 0, 0.5, out.data_ptr(), idx.data_ptr(), n.data_ptr(),
                       ws.data_ptr(), need, None)
    assert st == S.ERR_INVALID_ARG
    st = L.sffn_decode(x.data_ptr(), 1, w.ref(), 0, 0, 0.0, out.data_ptr(), idx.data_ptr(), n.data_ptr(),
                       ws.data_ptr(), need, None)
    assert st == S.OK
    torch.cuda.synchronize()
    # control block (int32 words): 0 error, 1 barrier arrivals (never reset),
    # 2 arrivals before the next call: one arrival per chunk CTA per call
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    R = -(-128 // min(sms, 128))
    C = -(-128 // R)  # chunks of d_ff = 128 neurons, one CTA each
    ctl = ws[:16].cpu().view(torch.int32).tolist()
    assert ctl[0] == 0 and ctl[1] == ctl[2] == C
    for _ in range(3):
        assert L.sffn_decode(x.data_ptr(), 1, w.ref(), 0, 0, 0.0, out.data_ptr(), idx.data_ptr(), n.data_ptr(),
                             ws.data_ptr(), need, None) == S.OK
    torch.cuda.synchronize()
    ctl2 = ws[:16].cpu().view(torch.int32).tolist()
    assert ctl2[1] == ctl2[2] == 4 * C
    assert S.read_device_error(ws) == 0
    assert not ws[:16].any()


@pytest.mark.gpu
def test_workspace_shared_between_entry_points(S):
    # one buffer serves token selection, prefill and decode in turn: the
    # control block stays valid whichever call used the buffer last
    from activation_sparse_ffn_gemv_gb300 import workloads as W
    d, F, L = 256, 512, 300
    layer = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in
             W.make_ffn_layer(5, seed=2, d_model=d, d_ff=F).items()}
    w = S.Weights(layer)
    need = max(S.workspace_size(S.WS_DECODE, 8, w), S.workspace_size(S.WS_SELECT, L, w),
               S.workspace_size(S.WS_PREFILL, L, w))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    X, Ya = (t.cuda() for t in W.make_prefill_inputs(L, d, seed=3))
    xt = W.make_tokens(5, 8, seed=4, d_model=d).cuda()
    ref_out, ref_idx, ref_n = S.decode(xt, w, S.MODE_EXACT)
    for _ in range(2):
        sel, n = S.token_select(Ya, 0.5, 16, 1, workspace=ws)
        S.prefill(X, Ya, w, sel, n, workspace=ws)
        o, i, nn = S.decode(xt, w, S.MODE_EXACT, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_out) and torch.equal(nn, ref_n)
        for b in range(8):
            k = int(nn[b])
            assert torch.equal(i[b, :k], ref_idx[b, :k])
    assert S.read_device_error(ws) == 0
