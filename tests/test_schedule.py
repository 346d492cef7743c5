"""The per-layer sparsity schedule of a multi-layer token-selective prefill
(host logic, no GPU): presets against the write-up's table, the three tiers,
and the stack driver's argument checks, which return before any CUDA call."""
from __future__ import annotations

import ctypes as C
import json
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "ffn_presets.json")


@pytest.fixture(scope="module")
def S():
    from activation_sparse_ffn_gemv_gb300 import build as B
    B.build()
    from activation_sparse_ffn_gemv_gb300 import sffn
    sffn.lib()
    return sffn


def test_presets_match_the_table(S):
    g = json.load(open(GOLDEN))
    for row in g["presets"]:
        s = S.schedule_preset(row["name"])
        assert s.dense_until == row["dense_until"], row["cite"]
        assert s.mass_thresh == pytest.approx(row["mass_thresh"], abs=1e-7), row["cite"]
        assert s.recent_n == row["recent_n"], row["cite"]
        assert s.min_keep == 1
        # the table names no deep tier
        assert s.deep_layer_start == 2**31 - 1 and s.mass_thresh_deep == s.mass_thresh
    d = g["demo_flags"]
    b = S.schedule_preset("balanced")
    assert (b.dense_until, b.recent_n) == (d["dense_until"], d["recent_n"])


def test_three_tiers(S):
    s = S.schedule(dense_until=2, mass_thresh=0.5, recent_n=16, deep_layer_start=5, mass_thresh_deep=0.2)
    got = [S.schedule_mass(s, l) for l in range(8)]
    assert got == pytest.approx([1.0, 1.0, 0.5, 0.5, 0.5, 0.2, 0.2, 0.2])
    # dense preset: every layer dense (mass 1 keeps every token)
    dn = S.schedule_preset("dense")
    assert all(S.schedule_mass(dn, l) == 1.0 for l in range(80))
    # deep tier starting before dense_until: shallow layers stay dense
    s2 = S.schedule(dense_until=4, mass_thresh=0.5, recent_n=0, deep_layer_start=2, mass_thresh_deep=0.3)
    assert [S.schedule_mass(s2, l) for l in range(6)] == pytest.approx([1, 1, 1, 1, 0.3, 0.3])


def test_invalid_schedules(S):
    ok = S.schedule(dense_until=1, mass_thresh=0.5, recent_n=4)
    assert S.schedule_mass(ok, -1) < 0
    for bad in (S.FFNSchedule(-1, 5, 0.5, 0.5, 4, 1), S.FFNSchedule(1, 5, -0.1, 0.5, 4, 1),
                S.FFNSchedule(1, 5, 0.5, -1.0, 4, 1), S.FFNSchedule(1, 5, 0.5, 0.5, -4, 1),
                S.FFNSchedule(1, 5, 0.5, 0.5, 4, 0)):
        assert S.schedule_mass(bad, 3) < 0
    with pytest.raises(S.SffnError):
        S.schedule_preset(7)


def test_layers_argument_checks_before_any_cuda_call(S):
    L = S.lib()
    w = S.FFNWeights(S.BF16, S.ACT_SILU, 64, 128, 16, 16, 16, None, None, None, None, None)
    ws = (S.FFNWeights * 2)(w, w)
    ya = (C.c_void_p * 2)(16, 16)
    s = S.schedule(dense_until=1, mass_thresh=0.5, recent_n=4)
    bad_s = S.FFNSchedule(1, 5, 0.5, 0.5, 4, 0)

    def call(x=16, ya_=ya, n=2, sched=s, out=32, L_=100, first=0):
        return L.sffn_prefill_layers(x, ya_, L_, n, ws, C.byref(sched), first, out, 16, 16, 256, 1 << 30, None)

    assert call(x=None) == S.ERR_INVALID_ARG
    assert call(ya_=None) == S.ERR_INVALID_ARG
    assert call(out=16) == S.ERR_INVALID_ARG          # x and out are the same buffer
    assert call(sched=bad_s) == S.ERR_INVALID_ARG
    assert call(first=-1) == S.ERR_INVALID_ARG
    assert call(n=0) == S.ERR_SHAPE
    assert call(L_=0) == S.ERR_SHAPE
    w2 = S.FFNWeights(S.BF16, S.ACT_SILU, 128, 128, 16, 16, 16, None, None, None, None, None)
    mixed = (S.FFNWeights * 2)(w, w2)
    assert L.sffn_prefill_layers(16, ya, 100, 2, mixed, C.byref(s), 0, 32, 16, 16, 256, 1 << 30,
                                 None) == S.ERR_SHAPE   # layers of different d_model
    need = L.sffn_prefill_layers_workspace_size(100, C.byref(w))
    assert need > 0
    assert L.sffn_prefill_layers(16, ya, 100, 2, ws, C.byref(s), 0, 32, 16, 16, 256, need - 1,
                                 None) == S.ERR_WORKSPACE
    assert L.sffn_prefill_layers_workspace_size(0, C.byref(w)) == 0
