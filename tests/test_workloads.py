"""The seeded input recipes against the workloads they stand in for (CPU).

Configs 1, 2 and 5 are pinned through the oracle's active fractions and the
mass-select closed form in test_oracle_pins.py; these pin the two recipes that
no oracle result depends on in a closed form: the log-normal W_down column
norms of the keep-ratio workload and the int4-g64 codes and scales.
"""
import math

import numpy as np
import pytest

from activation_sparse_ffn_gemv_gb300 import workloads as W


def _unpack_codes(packed: np.ndarray) -> np.ndarray:
    """Signed codes from the storage bytes (two's-complement nibbles, low nibble =
    even column)."""
    lo = (packed & 0xF).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    codes = np.empty((packed.shape[0], packed.shape[1] * 2), np.int16)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    return np.where(codes >= 8, codes - 16, codes)


def test_keep_ratio_down_column_norms_are_lognormal():
    # W_down[:, j] = N(0, 1/F)^d * exp(0.5 z_j): log ||W_down[:, j]|| =
    # 0.5 log(chi2_d / F) + 0.5 z_j, so its spread is sqrt(0.25 + 0.5 / d) (the
    # chi2 term, var(log chi2_d) ~ 2 / d) and its mean 0.5 (log(d / F) - 1 / d)
    c = W.CONFIGS[3]
    d, F = 256, c["d_ff"]
    layer = W.make_ffn_layer(3, seed=0, d_model=d)
    wdT = layer["w_downT"].float().numpy().astype(np.float64)
    ln = np.log(np.linalg.norm(wdT, axis=1))
    sig = c["down_col_lognormal"]
    want_sd = math.sqrt(sig * sig + 0.5 / d)
    want_mean = 0.5 * (math.log(d / F) - 1.0 / d)
    # standard errors over F = 11008 columns: 0.0034 (spread), 0.0048 (mean)
    assert abs(ln.std() - want_sd) < 0.015, (ln.std(), want_sd)
    assert abs(ln.mean() - want_mean) < 0.02, (ln.mean(), want_mean)
    # the gate and up rows carry no such factor
    wg = layer["w_gate"].float().numpy().astype(np.float64)
    assert np.log(np.linalg.norm(wg, axis=1)).std() < 0.1


def test_int4_codes_and_scales_follow_the_config():
    # codes uniform on {-8, ..., 7}; fp16 group scales U(0.005, 0.02), one per
    # 64 codes of a stored row
    d, F = 512, 2048
    layer = W.make_ffn_layer(4, seed=3, d_model=d, d_ff=F)
    for name in ("gate", "up", "downT"):
        packed = layer["w_" + name].numpy()
        assert packed.dtype == np.uint8 and packed.shape == (F, d // 2)
        codes = _unpack_codes(packed)
        assert codes.min() == -8 and codes.max() == 7
        counts = np.bincount((codes + 8).ravel(), minlength=16)
        n = codes.size
        chi2 = float(((counts - n / 16) ** 2 / (n / 16)).sum())
        assert chi2 < 50.0, chi2  # 15 degrees of freedom: P(chi2 > 50) < 1e-5
        s = layer["s_" + name].float().numpy()
        assert layer["s_" + name].dtype.is_floating_point and s.shape == (F, d // W.GROUP)
        assert s.min() >= 0.005 - 1e-5 and s.max() <= 0.02 + 1e-5
        # uniform: mean 0.0125 and the quartiles at 0.00875 / 0.01625
        assert abs(s.mean() - 0.0125) < 2e-4
        assert abs((s < 0.00875).mean() - 0.25) < 0.02
        assert abs((s < 0.01625).mean() - 0.75) < 0.02


def test_int4_storage_encoding_round_trips():
    import torch
    g = torch.Generator().manual_seed(7)
    codes = torch.randint(-8, 8, (5, 64), generator=g, dtype=torch.int8)
    back = _unpack_codes(W.pack_int4(codes).numpy())
    assert np.array_equal(back, codes.numpy().astype(np.int16))


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_decode_tokens_are_standard_normal(cfg):
    x = W.make_tokens(cfg, 64, seed=0, d_model=256).float().numpy().astype(np.float64)
    # 16384 draws: standard errors 0.008 (mean) and 0.0055 (spread)
    assert abs(x.mean()) < 0.04 and abs(x.std() - 1.0) < 0.03
    assert W.make_tokens(cfg, 1, seed=0).dtype == (W.torch.float32 if cfg == 1 else W.torch.bfloat16)
