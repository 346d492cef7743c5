"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds the input recipes only -- random draws, dtype casts and the
storage encoding of int4 codes -- and none of the FFN's arithmetic.  Both the
CUDA path and the fp64 oracle are fed from it.  The pages measure trained
models (ProSparse-Llama-2-7B, Qwen2.5-3B, Qwen3-32B) on text that is not
available here; these draws stand in for their shapes and sparsity:

1. tiny ReGLU decode      d=256,  F=688,   fp32, gate bias -1.0 (~15.9% active)
2. Llama-2-7B ReGLU decode d=4096, F=11008, bf16, gate bias ~N(-1.2, 0.3) (~12.5%)
3. Qwen2.5-3B SwiGLU       d=2048, F=11008, bf16, W_down columns x exp(0.5 z)
4. Qwen2.5-3B SwiGLU int4  same shape, symmetric int4 codes U{-8..7}, fp16 group
                           scales U(0.005, 0.02), group 64 along each stored row
5. token-selective prefill L=16384, d=5120, F=25600 bf16 SwiGLU,
                           Y_attn[t] = N(0,1) * exp(N(0,1))

Weights are N(0, 1/d_in) (d_in = d_model for W_gate/W_up, d_ff for W_down).
W_down is stored transposed, ``w_downT[j, :] = W_down[:, j]``, so that one
neuron's three weight vectors are contiguous rows.  Per-layer seed = seed + layer.
"""
from __future__ import annotations

import math

import torch

CONFIGS = {
    1: dict(name="tiny-reglu-decode", d_model=256, d_ff=688, wdtype="f32", act="relu",
            bias=("const", -1.0), tokens=64, batches=(1,), layers=1),
    2: dict(name="llama2-7b-reglu-decode", d_model=4096, d_ff=11008, wdtype="bf16", act="relu",
            bias=("normal", -1.2, 0.3), tokens=1024, batches=(1, 4, 8), layers=8),
    3: dict(name="qwen2.5-3b-swiglu-keep-ratio", d_model=2048, d_ff=11008, wdtype="bf16",
            act="silu", bias=None, down_col_lognormal=0.5, tokens=64, batches=(1,), layers=36,
            keep_M=(1, 2, 4, 8)),
    4: dict(name="qwen2.5-3b-swiglu-int4g64-sweep", d_model=2048, d_ff=11008, wdtype="int4_g64",
            act="silu", bias=None, tokens=64, batches=(1,), layers=36,
            sweep_a=(0.05, 0.1, 0.2, 0.4, 0.6, 0.8, 1.0)),
    5: dict(name="token-selective-prefill", L=16384, d_model=5120, d_ff=25600, wdtype="bf16",
            act="silu", bias=None, mass=(0.2, 0.5, 0.7, 1.0), recent_n=128, min_keep=1,
            token_scale_lognormal=1.0),
}

GROUP = 64


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, std, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def pack_int4(codes: torch.Tensor) -> torch.Tensor:
    """Storage encoding of signed codes in [-8, 7], [R, C] (C even) -> uint8
    [R, C/2]: two's-complement nibbles, low nibble = even column."""
    assert codes.dtype == torch.int8 and codes.shape[-1] % 2 == 0
    u = (codes.to(torch.int16) & 0xF).to(torch.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).contiguous()


def make_ffn_layer(cfg: int | dict, seed: int = 0, layer: int = 0, device="cpu",
                   d_model: int | None = None, d_ff: int | None = None,
                   wdtype: str | None = None, act: str | None = None) -> dict:
    """One FFN layer of a config.  Shapes/dtype may be overridden for small
    parity cases.  Returns tensors on ``device``:
    ``w_gate, w_up, w_downT`` ([F, d] fp32 / bf16, or packed int4 uint8 [F, d/2]),
    ``s_gate, s_up, s_downT`` (int4: fp16 [F, d/64], else None), ``b_gate``
    (fp32 [F] or None) and the metadata keys ``d_model, d_ff, wdtype, act``."""
    c = CONFIGS[cfg] if isinstance(cfg, int) else cfg
    d = int(d_model or c["d_model"])
    F = int(d_ff or c["d_ff"])
    wd = wdtype or c["wdtype"]
    a = act or c["act"]
    g = _gen(seed + layer, device)
    out = dict(d_model=d, d_ff=F, wdtype=wd, act=a, s_gate=None, s_up=None, s_downT=None,
               b_gate=None)
    if wd == "int4_g64":
        assert d % GROUP == 0
        for name in ("gate", "up", "downT"):
            codes = torch.randint(-8, 8, (F, d), generator=g, device=device, dtype=torch.int8)
            scales = (torch.rand((F, d // GROUP), generator=g, device=device) * 0.015 + 0.005)
            out["w_" + name] = pack_int4(codes)
            out["s_" + name] = scales.to(torch.float16).contiguous()
    else:
        dt = torch.float32 if wd == "f32" else torch.bfloat16
        wg = _normal((F, d), 1.0 / math.sqrt(d), g, device)
        wu = _normal((F, d), 1.0 / math.sqrt(d), g, device)
        wdT = _normal((F, d), 1.0 / math.sqrt(F), g, device)
        sig = c.get("down_col_lognormal")
        if sig:
            z = torch.randn((F, 1), generator=g, device=device)
            wdT = wdT * torch.exp(sig * z)
        out["w_gate"], out["w_up"], out["w_downT"] = (t.to(dt).contiguous() for t in (wg, wu, wdT))
    bias = c.get("bias")
    if bias is not None:
        if bias[0] == "const":
            out["b_gate"] = torch.full((F,), float(bias[1]), device=device, dtype=torch.float32)
        else:
            out["b_gate"] = (torch.randn((F,), generator=g, device=device) * bias[2] + bias[1]).contiguous()
    return out


def make_tokens(cfg: int | dict, n: int, seed: int = 0, device="cpu", d_model: int | None = None,
                xdtype: str | None = None) -> torch.Tensor:
    """Decode activations x [n, d] ~ N(0, 1): fp32 for the fp32 config, else bf16."""
    c = CONFIGS[cfg] if isinstance(cfg, int) else cfg
    d = int(d_model or c["d_model"])
    xd = xdtype or ("f32" if c["wdtype"] == "f32" else "bf16")
    g = _gen(10_000_019 + seed, device)
    x = torch.randn((n, d), generator=g, device=device)
    return (x if xd == "f32" else x.to(torch.bfloat16)).contiguous()


def make_prefill_inputs(L: int, d_model: int, seed: int = 0, device="cpu", sigma: float = 1.0,
                        zero_rows=None) -> tuple[torch.Tensor, torch.Tensor]:
    """X [L, d] ~ N(0,1) bf16 and Y_attn[t] = N(0,1) * exp(sigma * N(0,1)) bf16.
    ``zero_rows`` (optional index tensor) zeroes those attention-output rows."""
    g = _gen(20_000_003 + seed, device)
    X = torch.randn((L, d_model), generator=g, device=device).to(torch.bfloat16)
    s = torch.exp(sigma * torch.randn((L, 1), generator=g, device=device))
    Ya = torch.randn((L, d_model), generator=g, device=device) * s
    if zero_rows is not None:
        Ya[zero_rows] = 0.0
    return X.contiguous(), Ya.to(torch.bfloat16).contiguous()
