"""Pins for the fp64 oracle: each test ties an oracle function to something other
than itself -- a library routine on a special case, a closed form, brute force on
tiny inputs, or a value the pages print (tests/golden/).  CPU only."""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from activation_sparse_ffn_gemv_gb300 import workloads as W
from tests.oracle_io import dense_numpy, ffn_from_layer, mat_from_act

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def test_ieee_golden_bits():
    g = _golden("ieee_bits.json")
    for e in g["bf16_encode"]:
        v = eval(e["value"])  # arithmetic on literals only
        assert O.f64_to_bf16_bits(v) == int(e["bits"], 16), e
    for e in g["bf16_decode"]:
        assert O.bf16_to_f64(int(e["bits"], 16)) == eval(e["value"]), e
    for e in g["f16_decode"]:
        assert O.f16_to_f64(int(e["bits"], 16)) == eval(e["value"]), e


def test_int4_golden_dequant():
    g = _golden("ieee_bits.json")["int4_g64"]
    rows, cols = g["rows"], g["cols"]
    packed = np.zeros(rows * cols // 2, np.uint8)
    for i, b in enumerate(g["bytes_row0_head"]):
        packed[i] = int(b, 16)
    for i, b in enumerate(g["bytes_row1_head"]):
        packed[cols // 2 + i] = int(b, 16)
    scales = np.array([int(s, 16) for s in g["scales"]], np.uint16)
    m = O.Mat(O.INT4_G64, packed, rows, cols, scales=scales).to_f64()
    n0, n1 = len(g["expect_row0_head"]), len(g["expect_row1_head"])
    assert m[0, :n0].tolist() == g["expect_row0_head"]
    assert m[1, :n1].tolist() == g["expect_row1_head"]
    assert not m[0, n0:].any() and not m[1, n1:].any()


def test_f16_decode_all_patterns_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([O.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_all_patterns_vs_bitcast():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([O.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_rounding_vs_torch_on_float32_inputs():
    # torch rounds binary32 -> bf16 to nearest-even; on binary32 inputs a
    # direct fp64 -> bf16 rounding must agree exactly.
    g = torch.Generator().manual_seed(5)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 8)
    ties = (torch.randint(0, 1 << 16, (4000,), generator=g).to(torch.int32) << 16) | 0x8000
    x = torch.cat([x, ties.view(torch.float32)])
    x = x[torch.isfinite(x)]
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.f64_to_bf16_bits(float(v)) for v in x.numpy().astype(np.float64)], np.uint16)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# activations
# --------------------------------------------------------------------------

def test_activation_closed_forms():
    for z in (-7.5, -1.0, -1e-3, 0.0, 0.25, 3.0, 20.0):
        assert O.act(O.RELU, z) == max(z, 0.0)
        # SiLU(z) - SiLU(-z) = z * (sigmoid(z) + sigmoid(-z)) = z
        assert abs(O.act(O.SILU, z) - O.act(O.SILU, -z) - z) <= 1e-15 * max(1.0, abs(z))
    assert O.act(O.SILU, 0.0) == 0.0
    # sigmoid(ln 3) = 3/4
    assert abs(O.act(O.SILU, math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert abs(O.act(O.SILU, 40.0) - 40.0) < 1e-14


# --------------------------------------------------------------------------
# dense FFN special case = textbook GEMV chain (numpy fp64)
# --------------------------------------------------------------------------

CASES = [
    dict(wdtype="f32", act="relu", d_model=64, d_ff=40, bias=True),
    dict(wdtype="bf16", act="relu", d_model=128, d_ff=96, bias=True),
    dict(wdtype="bf16", act="silu", d_model=96, d_ff=72, bias=False),
    dict(wdtype="int4_g64", act="silu", d_model=128, d_ff=80, bias=False),
]


def _layer(case, seed=1):
    cfg = dict(W.CONFIGS[2 if case["bias"] else 3])
    cfg["down_col_lognormal"] = 0.5 if not case["bias"] else None
    return W.make_ffn_layer(cfg, seed=seed, d_model=case["d_model"], d_ff=case["d_ff"],
                            wdtype=case["wdtype"], act=case["act"])


def _x(case, n, seed=2):
    xd = "f32" if case["wdtype"] == "f32" else "bf16"
    return W.make_tokens(3, n, seed=seed, d_model=case["d_model"], xdtype=xd)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f'{c["wdtype"]}-{c["act"]}')
def test_dense_special_case_matches_numpy(case):
    layer, x = _layer(case), _x(case, 5)
    ffn = ffn_from_layer(layer)
    r = O.decode(ffn, mat_from_act(x), O.THRESHOLD, O.SCORE_GATE, 0.0)   # tau = 0 keeps all
    assert (r["n_active"] == case["d_ff"]).all()
    ref = dense_numpy(layer, x)
    err = np.linalg.norm(r["out"] - ref, axis=1) / np.linalg.norm(ref, axis=1)
    assert err.max() < 1e-12, err


@pytest.mark.parametrize("case", CASES, ids=lambda c: f'{c["wdtype"]}-{c["act"]}')
def test_keep_all_settings_equal_dense_bitwise(case):
    layer, x = _layer(case), _x(case, 4)
    ffn, xm = ffn_from_layer(layer), mat_from_act(x)
    dense = O.decode(ffn, xm, O.THRESHOLD, O.SCORE_GATE, 0.0)["out"]
    for sk in (O.SCORE_GATE, O.SCORE_GATE_UP):
        r = O.decode(ffn, xm, O.KEEP_RATIO, sk, 1.0)      # tier M = 1 keeps everything
        assert np.array_equal(r["out"], dense)
        assert (r["n_active"] == case["d_ff"]).all()
    if case["act"] == "relu":
        # exact ReLU gating skips only zero activations: same output, bit for bit
        r = O.decode(ffn, xm, O.EXACT)
        assert np.array_equal(r["out"], dense)
        assert (r["n_active"] < case["d_ff"]).all()


def test_exact_set_is_positive_gate():
    case = CASES[1]
    layer, x = _layer(case), _x(case, 6)
    r = O.decode(ffn_from_layer(layer), mat_from_act(x), O.EXACT, details=True)
    Wg = ffn_from_layer(layer).w_gate.to_f64()
    G = mat_from_act(x).to_f64() @ Wg.T + layer["b_gate"].double().numpy()
    for b in range(x.shape[0]):
        want = np.flatnonzero(G[b] > 0)
        assert np.array_equal(r["active_idx"][b, : r["n_active"][b]], want)
        assert np.all(r["cond"][b] >= np.abs(r["g"][b]) * (1 - 1e-12))


# --------------------------------------------------------------------------
# weight-aware score, threshold and keep-ratio selection
# --------------------------------------------------------------------------

def _closed_form_layer(g_vals, col_scale, u_vals, d):
    """x = e_0; W_gate[j] = g_j e_0 -> g = g_vals exactly; W_up[j] = u_j e_0;
    W_downT[j] = c_j e_(j mod d) -> ||W_down[:, j]||_2 = |c_j|."""
    F = len(g_vals)
    wg = np.zeros((F, d), np.float32)
    wu = np.zeros((F, d), np.float32)
    wd = np.zeros((F, d), np.float32)
    wg[:, 0] = g_vals
    wu[:, 0] = u_vals
    wd[np.arange(F), np.arange(F) % d] = col_scale
    x = np.zeros((1, d), np.float32)
    x[0, 0] = 1.0
    return wg, wu, wd, x


@pytest.mark.parametrize("act", [O.RELU, O.SILU])
def test_score_closed_form(act):
    rng = np.random.default_rng(3)
    F, d = 24, 8
    g = rng.choice(np.arange(-12, 13), F, replace=True).astype(np.float32) / 4
    c = rng.choice([0.25, 0.5, 1.0, 2.0, 4.0], F).astype(np.float32)
    u = rng.choice([-3.0, -1.0, 0.5, 2.0], F).astype(np.float32)
    wg, wu, wd, x = _closed_form_layer(g, c, u, d)
    ffn = O.FFN(O.Mat(O.F32, wg, F, d), O.Mat(O.F32, wu, F, d), O.Mat(O.F32, wd, F, d), act)
    xm = O.Mat(O.F32, x, 1, d)
    a = np.array([max(v, 0.0) if act == O.RELU else v / (1 + math.exp(-v)) for v in g.astype(float)])
    r = O.decode(ffn, xm, O.THRESHOLD, O.SCORE_GATE, 0.0, details=True)
    assert np.array_equal(r["norms"], np.abs(c).astype(float))
    assert np.allclose(r["score"][0], np.abs(a) * c, rtol=1e-15, atol=0)
    assert np.array_equal(r["u"][0], u.astype(float))
    r2 = O.decode(ffn, xm, O.THRESHOLD, O.SCORE_GATE_UP, 0.0, details=True)
    assert np.allclose(r2["score"][0], np.abs(a * u) * c, rtol=1e-15, atol=0)
    # threshold keeps exactly {score >= tau}, the cut itself included
    tau = float(np.sort(r["score"][0])[F // 2])
    r3 = O.decode(ffn, xm, O.THRESHOLD, O.SCORE_GATE, tau, details=True)
    want = np.flatnonzero(r["score"][0] >= tau)
    assert np.array_equal(r3["active_idx"][0, : r3["n_active"][0]], want)
    # the output on a known set is the sum of h_j * W_down[:, j] over that set
    h = a * u
    ref = np.zeros(d)
    for j in want:
        ref[j % d] += h[j] * c[j]
    assert np.allclose(r3["out"][0], ref, rtol=1e-15, atol=1e-300)


def test_silu_slope_bound_behind_the_tie_band():
    # The oracle scales the tie band of an activation-based score by 1.1: an
    # error e in g moves act(g) by at most max|act'| * e.  ReLU's slope is at most
    # 1; SiLU's, s(z) (1 + z (1 - s(z))), peaks near z = 2.3994 at 1.09984.
    z = np.linspace(-20.0, 20.0, 4_000_001)
    sg = 1.0 / (1.0 + np.exp(-z))
    slope = sg * (1.0 + z * (1.0 - sg))
    assert 1.0998 < slope.max() < 1.1
    assert abs(z[slope.argmax()] - 2.3994) < 1e-3
    assert slope.min() > -0.1   # the negative dip is shallower than the bound too


@pytest.mark.parametrize("act", [O.RELU, O.SILU])
def test_tie_band_conditioning_closed_form(act):
    # One-hot rows make every dot product a single exact term, so the
    # conditioning sums are closed forms: cg = |g_j - b_j| + |b_j|, cu = |u_j|.
    # The bound is tight there (a one-term dot has relative error exactly one
    # rounding of its only term).  Exact gating: cond = cg.  GATE score:
    # cond = 1.1 cg n_j.  GATE_UP score: cond = (|u| 1.1 cg + max(|a|, cg) cu) n_j,
    # the first-order error of |a u| n with a's error bounded through the slope
    # and max(|a|, cg) covering a near 0.
    rng = np.random.default_rng(8)
    F, d = 16, 8
    g = rng.choice(np.arange(-12, 13), F).astype(np.float32) / 4
    c = rng.choice([0.25, 0.5, 1.0, 2.0], F).astype(np.float32)
    u = rng.choice([-3.0, -1.0, 0.5, 2.0], F).astype(np.float32)
    b = rng.choice([-0.5, 0.0, 0.25], F).astype(np.float32)
    wg, wu, wd, x = _closed_form_layer(g, c, u, d)
    ffn = O.FFN(O.Mat(O.F32, wg, F, d), O.Mat(O.F32, wu, F, d), O.Mat(O.F32, wd, F, d), act, torch.from_numpy(b))
    xm = O.Mat(O.F32, x, 1, d)
    gg = g.astype(float) + b.astype(float)
    a = np.maximum(gg, 0.0) if act == O.RELU else gg / (1.0 + np.exp(-gg))
    cg = np.abs(g.astype(float)) + np.abs(b.astype(float))
    cu = np.abs(u.astype(float))
    n = np.abs(c.astype(float))
    r = O.decode(ffn, xm, O.EXACT, details=True)
    assert np.array_equal(r["cond"][0], cg)
    r = O.decode(ffn, xm, O.THRESHOLD, O.SCORE_GATE, 0.0, details=True)
    assert np.allclose(r["cond"][0], 1.1 * cg * n, rtol=1e-15, atol=0)
    r = O.decode(ffn, xm, O.THRESHOLD, O.SCORE_GATE_UP, 0.0, details=True)
    want = (np.abs(u.astype(float)) * 1.1 * cg + np.maximum(np.abs(a), cg) * cu) * n
    assert np.allclose(r["cond"][0], want, rtol=1e-15, atol=0)


def test_keep_ratio_bruteforce_small():
    rng = np.random.default_rng(11)
    for trial in range(30):
        F = int(rng.integers(2, 13))
        d = 64
        layer = W.make_ffn_layer(W.CONFIGS[3], seed=100 + trial, d_model=d, d_ff=F,
                                 wdtype="bf16", act="silu")
        x = W.make_tokens(3, 1, seed=trial, d_model=d)
        ffn, xm = ffn_from_layer(layer), mat_from_act(x)
        for sk in (O.SCORE_GATE, O.SCORE_GATE_UP):
            ratio = float(rng.uniform(0.01, 1.0))
            r = O.decode(ffn, xm, O.KEEP_RATIO, sk, ratio, details=True)
            s = r["score"][0]
            k = max(1, int(math.floor(F * ratio)))
            assert r["n_active"][0] == k == O.keep_count(F, ratio)
            best = max(itertools.combinations(range(F), k), key=lambda S: sum(s[list(S)]))
            assert tuple(r["active_idx"][0, :k]) == best


def test_keep_ratio_ties_go_to_lower_index():
    F, d = 10, 8
    g = np.array([1, 2, 2, 2, 3, 0.5, 2, 3, 1, 2], np.float32)
    wg, wu, wd, x = _closed_form_layer(g, np.ones(F, np.float32), np.ones(F, np.float32), d)
    ffn = O.FFN(O.Mat(O.F32, wg, F, d), O.Mat(O.F32, wu, F, d), O.Mat(O.F32, wd, F, d), O.RELU)
    r = O.decode(ffn, O.Mat(O.F32, x, 1, d), O.KEEP_RATIO, O.SCORE_GATE, 0.45)   # k = 4
    assert r["active_idx"][0, :4].tolist() == [1, 2, 4, 7]


def test_keep_count_tiers():
    # tier M keeps F/M: exact for F = 11008 and M in {1, 2, 4, 8}
    for M, k in ((1, 11008), (2, 5504), (4, 2752), (8, 1376)):
        assert O.keep_count(11008, 1.0 / M) == k
    assert O.keep_count(5, 1e-6) == 1          # max(1, .)


# --------------------------------------------------------------------------
# byte model (denseflux) -- printed worked values
# --------------------------------------------------------------------------

def test_byte_model_exact_and_printed_pairs():
    for fmt, d in ((O.F32, 256), (O.BF16, 4096), (O.INT4_G64, 2048)):
        F = 11008
        dense = O.bytes_kept(fmt, d, F, O.SCORE_GATE, F)
        assert dense == 3 * F * O.row_bytes(fmt, d)
        for n in (0, 1, 1376, 5000, F):
            a = n / F
            assert abs(O.bytes_kept(fmt, d, F, O.SCORE_GATE, n) / dense - (1 + 2 * a) / 3) < 1e-15
            assert abs(O.bytes_kept(fmt, d, F, O.SCORE_GATE_UP, n) / dense - (2 + a) / 3) < 1e-15
    assert O.row_bytes(O.INT4_G64, 2048) == 1024 + 64
    g = _golden("byte_model.json")
    F = 100000
    for e in g["kept_fraction"]:
        n = round(e["a"] * F)
        r = O.bytes_kept(O.BF16, 64, F, O.SCORE_GATE, n) / O.bytes_kept(O.BF16, 64, F, O.SCORE_GATE, F)
        assert abs(r - e["kept"]) <= e["abs_tol"], e
    for e in g["skip_saving"]:
        n = round((1 - e["skipped"]) * F)
        r = 1 - O.bytes_kept(O.BF16, 64, F, O.SCORE_GATE, n) / O.bytes_kept(O.BF16, 64, F, O.SCORE_GATE, F)
        assert abs(r - e["saved"]) <= e["abs_tol"], e
    for e in g["ideal_speedup"]:
        n = round(e["a"] * F)
        ideal = O.bytes_kept(O.BF16, 64, F, O.SCORE_GATE, F) / O.bytes_kept(O.BF16, 64, F, O.SCORE_GATE, n)
        assert abs(ideal - e["ideal"]) <= 1e-12
        assert abs(e["measured"] / ideal - e["fraction_of_ideal"]) <= e["abs_tol"]
    for e in g["ffn_share"]:
        ffn_params = O.bytes_kept(O.BF16, e["d_model"], e["d_ff"], O.SCORE_GATE, e["d_ff"]) / 2
        assert ffn_params == e["ffn_params"]
        assert abs(ffn_params / (ffn_params + e["attn_params"]) - 2 / 3) < 0.01


# --------------------------------------------------------------------------
# synthetic active fractions (generator + gate together)
# --------------------------------------------------------------------------

def _phi_upper(z):
    return 0.5 * math.erfc(z / math.sqrt(2))


def test_active_fraction_tiny_reglu():
    # g = W_gate x - 1 with W_gate x ~ N(0, 1): P(g > 0) = P(N(0,1) > 1)
    layer = W.make_ffn_layer(1, seed=0)
    x = W.make_tokens(1, 64, seed=0)
    r = O.decode(ffn_from_layer(layer), mat_from_act(x), O.EXACT, nthreads=4)
    frac = r["n_active"].mean() / layer["d_ff"]
    assert abs(frac - _phi_upper(1.0)) < 0.01, frac


def test_active_fraction_llama_reglu_shape():
    # b ~ N(-1.2, 0.3): g ~ N(-1.2, 1 + 0.09) -> P(g > 0) = P(N(0,1) > 1.2 / sqrt(1.09))
    layer = W.make_ffn_layer(2, seed=0)
    x = W.make_tokens(2, 4, seed=0)
    r = O.decode(ffn_from_layer(layer), mat_from_act(x), O.EXACT, nthreads=os.cpu_count() or 1)
    frac = r["n_active"].mean() / layer["d_ff"]
    assert abs(frac - _phi_upper(1.2 / math.sqrt(1.09))) < 0.01, frac


# --------------------------------------------------------------------------
# token selection (RedKnot)
# --------------------------------------------------------------------------

def test_token_norms_closed_form():
    d = 64
    y = np.zeros((4, d), np.float32)
    y[0, :2] = (3.0, 4.0)                  # 5
    y[1, :] = -0.5                         # 0.5 * sqrt(64) = 4
    y[3, 7] = -2.0                         # 2
    ybf = torch.from_numpy(y).to(torch.bfloat16)
    s = O.token_norms(mat_from_act(ybf))
    assert s.tolist() == [5.0, 4.0, 0.0, 2.0]


def _bruteforce_prefix(s, m):
    """Minimum-cardinality subset with mass >= m * total, then maximum mass."""
    L = len(s)
    T = float(np.sum(s))
    best = None
    for k in range(0, L + 1):
        for S in itertools.combinations(range(L), k):
            mass = float(np.sum(s[list(S)])) if S else 0.0
            if mass >= m * T and (best is None or mass > best[1]):
                best = (S, mass)
        if best is not None:
            return set(best[0])
    return set(range(L))


def test_mass_select_bruteforce_small():
    rng = np.random.default_rng(7)
    for trial in range(60):
        L = int(rng.integers(1, 12))
        s = rng.lognormal(0, 1, L)
        m = float(rng.choice([1e-9, 0.1, 0.2, 0.5, 0.7, 0.95, 0.999]))
        sel, pre = O.mass_select(s, m, recent_n=0, min_keep=1)
        assert set(pre.tolist()) == _bruteforce_prefix(s, m), (s, m)
        assert set(sel.tolist()) == set(pre.tolist()) or len(pre) == 0


def test_mass_select_guards():
    rng = np.random.default_rng(9)
    for trial in range(200):
        L = int(rng.integers(1, 300))
        s = rng.lognormal(0, 1.0, L)
        if trial % 7 == 0:
            s[rng.integers(0, L, L // 2)] = 0.0
        m = float(rng.choice([0.0, 1e-9, 0.2, 0.5, 0.7, 0.99, 1.0, 1.5]))
        recent = int(rng.choice([0, 1, 5, 128, 1000]))
        min_keep = int(rng.choice([1, 2, 17, 500]))
        sel, pre = O.mass_select(s, m, recent, min_keep)
        S = set(sel.tolist())
        assert np.all(np.diff(sel) > 0)
        assert set(range(max(0, L - recent), L)) <= S
        assert len(S) >= min(min_keep, L)
        assert set(pre.tolist()) <= S
        if m >= 1.0:
            assert len(S) == L
        if m <= 0.0:
            assert len(pre) == 0
    # all-zero importances fall back to dense
    sel, _ = O.mass_select(np.zeros(50), 0.3, 4, 1)
    assert sel.tolist() == list(range(50))
    # ties: equal importances are taken in index order
    sel, pre = O.mass_select(np.ones(10), 0.25, 0, 1)
    assert pre.tolist() == [0, 1, 2]


def test_mass_select_lognormal_fraction():
    """Closed form: for s = exp(sigma Z), the smallest top set holding a fraction
    m of the total mass is a fraction Phi(Phi^-1(m) - sigma) of the tokens."""
    from statistics import NormalDist
    c = W.CONFIGS[5]
    L, d = c["L"], c["d_model"]
    _, Ya = W.make_prefill_inputs(L, d, seed=0)
    s = O.token_norms(mat_from_act(Ya))
    N = NormalDist()
    for m in (0.2, 0.5, 0.7):
        _, pre = O.mass_select(s, m, 0, 1)
        want = N.cdf(N.inv_cdf(m) - c["token_scale_lognormal"])
        assert abs(len(pre) / L - want) < 0.01, (m, len(pre) / L, want)


# --------------------------------------------------------------------------
# prefill rows
# --------------------------------------------------------------------------

def test_residual_rounding():
    X = torch.tensor([[1.0, 1.0, -3.0, 0.0]], dtype=torch.bfloat16)
    Ya = torch.tensor([[2 ** -8, 3 * 2 ** -8, 3.0, -0.0]], dtype=torch.bfloat16)
    y = O.residual(mat_from_act(X), mat_from_act(Ya))
    # 1 + 2^-8 ties to 1.0; 1 + 3*2^-8 ties to 1 + 2^-6; -3 + 3 = +0
    assert y[0].tolist() == [0x3F80, 0x3F82, 0x0000, 0x0000]
    g = torch.Generator().manual_seed(1)
    X = torch.randn(64, 256, generator=g).to(torch.bfloat16)
    Ya = (torch.randn(64, 256, generator=g) * 3).to(torch.bfloat16)
    exact = X.double() + Ya.double()
    ok = (exact.float().double() == exact)      # the binary32 sum is exact here
    want = (X.float() + Ya.float()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.residual(mat_from_act(X), mat_from_act(Ya))
    assert ok.float().mean() > 0.99
    assert np.array_equal(got[ok.numpy()], want[ok.numpy()])


def test_prefill_rows_match_numpy_dense_ffn():
    L, d, F = 24, 64, 96
    layer = W.make_ffn_layer(5, seed=4, d_model=d, d_ff=F)
    X, Ya = W.make_prefill_inputs(L, d, seed=4)
    ffn = ffn_from_layer(layer)
    Xm, Yam = mat_from_act(X), mat_from_act(Ya)
    mask = np.zeros(L, np.uint8)
    mask[::3] = 1
    rows = np.arange(L, dtype=np.int32)
    z, out = O.prefill_rows(ffn, Xm, Yam, mask, rows, nthreads=2)
    Ybits = O.residual(Xm, Yam)
    Y = torch.from_numpy(Ybits.view(np.int16)).view(torch.bfloat16)
    ref = dense_numpy(layer, Y)
    sel = mask.astype(bool)
    assert np.allclose(z[sel], ref[sel], rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert not z[~sel].any()
    assert np.array_equal(out[~sel], Ybits[~sel])
    want = np.array([[O.f64_to_bf16_bits(v) for v in row] for row in
                     (Y.double().numpy()[sel] + ref[sel])], np.uint16)
    # identical except where the fp64 rounding of y + z lands on a bf16 tie boundary
    assert (out[sel] != want).mean() < 1e-3
