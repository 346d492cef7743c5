"""Adapters from seeded workload tensors (CPU) to the oracle's stored matrices."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

_FMT = {"f32": O.F32, "bf16": O.BF16, "int4_g64": O.INT4_G64}
_ACT = {"relu": O.RELU, "silu": O.SILU}


def mat_from_weight(layer: dict, name: str) -> O.Mat:
    F, d, wd = layer["d_ff"], layer["d_model"], layer["wdtype"]
    w = layer["w_" + name].cpu()
    if wd == "int4_g64":
        return O.Mat(O.INT4_G64, w, F, d, scales=layer["s_" + name].cpu())
    return O.Mat(_FMT[wd], w, F, d)


def ffn_from_layer(layer: dict) -> O.FFN:
    b = layer.get("b_gate")
    return O.FFN(mat_from_weight(layer, "gate"), mat_from_weight(layer, "up"),
                 mat_from_weight(layer, "downT"), _ACT[layer["act"]],
                 None if b is None else b.cpu())


def mat_from_act(x: torch.Tensor) -> O.Mat:
    x = x.cpu().contiguous()
    fmt = O.F32 if x.dtype == torch.float32 else O.BF16
    return O.Mat(fmt, x, x.shape[0], x.shape[1])


def dense_numpy(layer: dict, x: torch.Tensor) -> np.ndarray:
    """Textbook dense gated FFN in numpy fp64 on the exactly dequantised weights:
    W_down @ (act(W_gate @ x + b) * (W_up @ x)), one column per token."""
    Wg = mat_from_weight(layer, "gate").to_f64()
    Wu = mat_from_weight(layer, "up").to_f64()
    Wd = mat_from_weight(layer, "downT").to_f64().T          # W_down [d, F]
    X = mat_from_act(x).to_f64().T                            # [d, B]
    G = Wg @ X
    if layer.get("b_gate") is not None:
        G = G + layer["b_gate"].double().numpy()[:, None]
    if layer["act"] == "relu":
        A = np.maximum(G, 0.0)
    else:
        A = G * (1.0 / (1.0 + np.exp(-G)))
    return (Wd @ (A * (Wu @ X))).T
