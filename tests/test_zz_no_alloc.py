"""sffn_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (they receive their buffers from a framework or plugin host and
have no allocator, or may not allocate while serving), so they cannot pass the
workspace sffn_decode needs.  The call uses a fixed scratch array inside the
library instead.

Checked here through the C ABI: two calls in a row (different shapes and modes,
so the second one runs on scratch the first one left behind) each give exactly
the outputs of sffn_decode with a caller workspace (the same kernels, so the
same bits), the array's error word reads back clear, and a request larger than
the array is rejected.  This file is collected last on purpose."""
from __future__ import annotations

import ctypes as C

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


def _call_noalloc(S, x, w, mode, score, param):
    B = x.shape[0]
    out = torch.full_like(x, float("nan"))
    idx = torch.full((B, w.d_ff), -1, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    st = S.lib().sffn_decode_noalloc(x.data_ptr(), B, w.ref(), mode, score, C.c_float(param), out.data_ptr(),
                                     idx.data_ptr(), n.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == S.OK, S.status_string(st)
    return out, idx, n


def _compare(S, layer_cpu, x_cpu, mode, score, param):
    layer = layer_to(layer_cpu, "cuda")
    w = S.Weights(layer)
    if mode != S.MODE_EXACT:
        w.set_down_norms(S.down_norms(w))
    x = x_cpu.cuda()
    assert S.workspace_size(S.WS_DECODE, x.shape[0], w) <= S.NOALLOC_SCRATCH_BYTES
    ref_out, ref_idx, ref_n = S.decode(x, w, mode, score, param)
    out, idx, n = _call_noalloc(S, x, w, mode, score, param)
    torch.cuda.synchronize()
    assert torch.equal(n, ref_n)
    for b in range(x.shape[0]):
        k = int(n[b])
        assert torch.equal(idx[b, :k], ref_idx[b, :k])
    # the partial sums are added in a fixed order: the outputs are bit-identical
    assert torch.equal(out.view(torch.int16) if out.dtype == torch.bfloat16 else out,
                       ref_out.view(torch.int16) if ref_out.dtype == torch.bfloat16 else ref_out)


def test_noalloc_matches_workspace_decode_two_calls(S):
    # call 1: Llama-2-7B-shaped ReGLU FFN, exact gating, one token
    _compare(S, W.make_ffn_layer(2, seed=5), W.make_tokens(2, 1, seed=5), S.MODE_EXACT, S.SCORE_GATE, 0.0)
    # call 2: Qwen2.5-3B-shaped SwiGLU FFN, keep-ratio 1/4 with the gate-and-up score, two tokens
    _compare(S, W.make_ffn_layer(3, seed=6), W.make_tokens(3, 2, seed=6), S.MODE_KEEP_RATIO,
             S.SCORE_GATE_UP, 0.25)
    # no bounded wait gave up in either call
    assert S.decode_noalloc_read_error() == 0


def test_noalloc_rejects_requests_beyond_the_array(S):
    layer = layer_to(W.make_ffn_layer(2, seed=7), "cuda")
    w = S.Weights(layer)
    x = W.make_tokens(2, 8, seed=7).cuda()
    assert S.workspace_size(S.WS_DECODE, 8, w) > S.NOALLOC_SCRATCH_BYTES
    out = torch.empty_like(x)
    idx = torch.empty((8, w.d_ff), dtype=torch.int32, device="cuda")
    n = torch.empty(8, dtype=torch.int32, device="cuda")
    st = S.lib().sffn_decode_noalloc(x.data_ptr(), 8, w.ref(), S.MODE_EXACT, S.SCORE_GATE, C.c_float(0.0),
                                     out.data_ptr(), idx.data_ptr(), n.data_ptr(), None)
    assert st == S.ERR_WORKSPACE
