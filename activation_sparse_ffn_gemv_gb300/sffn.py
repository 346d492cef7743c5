"""ctypes binding over libsffn.so (include/sffn.h) -- argument marshalling only.

PyTorch supplies device memory and streams: tensors are passed as raw device
pointers and the current torch stream is the launch stream.  Every step of the
computation runs in the library's CUDA kernels; if the library has not been
built (``__graft_entry__.build()`` or ``python -m
activation_sparse_ffn_gemv_gb300.build``) the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsffn.so")

# enums (include/sffn.h)
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(9)
MODE_EXACT, MODE_THRESHOLD, MODE_KEEP_RATIO = 0, 1, 2
ACT_RELU, ACT_SILU = 0, 1
F32, BF16, INT4_G64 = 0, 1, 2
SCORE_GATE, SCORE_GATE_UP = 0, 1
WS_DECODE, WS_SELECT, WS_PREFILL = 0, 1, 2
PRESET_SPEED, PRESET_BALANCED, PRESET_QUALITY, PRESET_DENSE = 0, 1, 2, 3
_PRESET = {"speed": PRESET_SPEED, "balanced": PRESET_BALANCED, "quality": PRESET_QUALITY, "dense": PRESET_DENSE}
NOALLOC_SCRATCH_BYTES = 4 << 20

_WDTYPE = {"f32": F32, "bf16": BF16, "int4_g64": INT4_G64}
_ACT = {"relu": ACT_RELU, "silu": ACT_SILU}


class SffnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class FFNWeights(C.Structure):
    _fields_ = [("wdtype", C.c_int32), ("act", C.c_int32), ("d_model", C.c_int32), ("d_ff", C.c_int32),
                ("w_gate", C.c_void_p), ("w_up", C.c_void_p), ("w_downT", C.c_void_p),
                ("s_gate", C.c_void_p), ("s_up", C.c_void_p), ("s_downT", C.c_void_p),
                ("b_gate", C.c_void_p), ("down_norms", C.c_void_p)]


class FFNSchedule(C.Structure):
    _fields_ = [("dense_until", C.c_int32), ("deep_layer_start", C.c_int32), ("mass_thresh", C.c_float),
                ("mass_thresh_deep", C.c_float), ("recent_n", C.c_int32), ("min_keep", C.c_int32)]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libsffn.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        P, I, F, S = C.c_void_p, C.c_int, C.c_float, C.c_size_t
        W = C.POINTER(FFNWeights)
        L.sffn_status_string.argtypes = [I]
        L.sffn_status_string.restype = C.c_char_p
        L.sffn_workspace_size.argtypes = [I, I, W]
        L.sffn_workspace_size.restype = S
        L.sffn_down_norms.argtypes = [W, P, P]
        L.sffn_down_norms.restype = I
        L.sffn_decode.argtypes = [P, I, W, I, I, F, P, P, P, P, S, P]
        L.sffn_decode.restype = I
        L.sffn_decode_dense.argtypes = [P, I, W, P, P, S, P]
        L.sffn_decode_dense.restype = I
        L.sffn_decode_predicted.argtypes = [P, W, P, P, I, F, P, P, P, P, S, P]
        L.sffn_decode_predicted.restype = I
        L.sffn_decode_tiered.argtypes = [P, I, W, I, F, P, I, P, P, P, P, S, P]
        L.sffn_decode_tiered.restype = I
        L.sffn_tier_core_workspace_size.argtypes = [I, I]
        L.sffn_tier_core_workspace_size.restype = S
        L.sffn_tier_core_set.argtypes = [P, I, I, I, I, P, P, S, P]
        L.sffn_tier_core_set.restype = I
        L.sffn_moe_progressive_k.argtypes = [I]
        L.sffn_moe_progressive_k.restype = I
        L.sffn_moe_route.argtypes = [P, I, I, I, F, C.POINTER(C.c_int32), I, I, P, P, P, P]
        L.sffn_moe_route.restype = I
        L.sffn_moe_budget_workspace_size.argtypes = [I, I]
        L.sffn_moe_budget_workspace_size.restype = S
        L.sffn_moe_block_budget.argtypes = [P, I, I, F, F, F, I, P, P, P, P, P, S, P]
        L.sffn_moe_block_budget.restype = I
        L.sffn_gate_scores.argtypes = [P, I, W, I, P, P, S, P]
        L.sffn_gate_scores.restype = I
        L.sffn_token_select.argtypes = [P, I, I, F, I, I, P, P, P, S, P]
        L.sffn_token_select.restype = I
        L.sffn_prefill.argtypes = [P, P, I, W, P, P, P, P, S, P]
        L.sffn_prefill.restype = I
        L.sffn_decode_noalloc.argtypes = [P, I, W, I, I, F, P, P, P, P]
        L.sffn_decode_noalloc.restype = I
        L.sffn_decode_noalloc_read_error.argtypes = [C.POINTER(C.c_int32), P]
        L.sffn_decode_noalloc_read_error.restype = I
        L.sffn_read_device_error.argtypes = [P, C.POINTER(C.c_int32), P]
        L.sffn_read_device_error.restype = I
        SP = C.POINTER(FFNSchedule)
        L.sffn_schedule_preset.argtypes = [I, SP]
        L.sffn_schedule_preset.restype = I
        L.sffn_schedule_mass.argtypes = [SP, I]
        L.sffn_schedule_mass.restype = F
        L.sffn_prefill_layers_workspace_size.argtypes = [I, W]
        L.sffn_prefill_layers_workspace_size.restype = S
        L.sffn_prefill_layers.argtypes = [P, C.POINTER(C.c_void_p), I, I, W, SP, I, P, P, P, P, S, P]
        L.sffn_prefill_layers.restype = I
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().sffn_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != OK:
        raise SffnError(st, where)


class Weights:
    """One FFN layer on the device: keeps the tensors alive and the C struct."""

    def __init__(self, layer: dict, down_norms: torch.Tensor | None = None):
        self.layer = layer
        self.d_model, self.d_ff = int(layer["d_model"]), int(layer["d_ff"])
        self.wdtype, self.act = layer["wdtype"], layer["act"]
        self.down_norms = down_norms
        self.c = FFNWeights(_WDTYPE[self.wdtype], _ACT[self.act], self.d_model, self.d_ff,
                            _ptr(layer["w_gate"]), _ptr(layer["w_up"]), _ptr(layer["w_downT"]),
                            _ptr(layer.get("s_gate")), _ptr(layer.get("s_up")), _ptr(layer.get("s_downT")),
                            _ptr(layer.get("b_gate")), _ptr(down_norms))

    def set_down_norms(self, norms: torch.Tensor):
        self.down_norms = norms
        self.c.down_norms = _ptr(norms)

    def ref(self):
        return C.byref(self.c)


def workspace_size(which: int, n: int, w: Weights | None) -> int:
    return int(lib().sffn_workspace_size(int(which), int(n), None if w is None else w.ref()))


def alloc_workspace(which: int, n: int, w: Weights | None, device=None) -> torch.Tensor:
    nbytes = workspace_size(which, n, w)
    if nbytes == 0:
        raise SffnError(ERR_INVALID_ARG, "workspace_size")
    # torch's caching allocator returns >= 512-byte aligned blocks
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def down_norms(w: Weights, norms: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if norms is None:
        norms = torch.empty(w.d_ff, dtype=torch.float32, device="cuda")
    _check(lib().sffn_down_norms(w.ref(), _ptr(norms), _stream(stream)), "sffn_down_norms")
    return norms


def decode(x: torch.Tensor, w: Weights, mode: int, score: int = SCORE_GATE, param: float = 0.0,
           out=None, active_idx=None, n_active=None, workspace=None, stream=None):
    """Returns (out [B, d], active_idx [B, d_ff] int32, n_active [B] int32)."""
    B = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    if active_idx is None:
        active_idx = torch.empty((B, w.d_ff), dtype=torch.int32, device=x.device)
    if n_active is None:
        n_active = torch.empty(B, dtype=torch.int32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(WS_DECODE, B, w, x.device)
    st = lib().sffn_decode(_ptr(x), B, w.ref(), int(mode), int(score), float(param), _ptr(out),
                           _ptr(active_idx), _ptr(n_active), _ptr(workspace), workspace.numel(),
                           _stream(stream))
    _check(st, "sffn_decode")
    return out, active_idx, n_active


def decode_dense(x: torch.Tensor, w: Weights, out=None, workspace=None, stream=None):
    """The dense layer (every neuron): out [B, d]."""
    B = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    if workspace is None:
        workspace = alloc_workspace(WS_DECODE, B, w, x.device)
    st = lib().sffn_decode_dense(_ptr(x), B, w.ref(), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sffn_decode_dense")
    return out


def decode_predicted(x: torch.Tensor, w: Weights, factor_a, factor_b, alpha: float, out=None, active_idx=None,
                     n_active=None, workspace=None, stream=None):
    """One token with the low-rank gate predictor: factor_a [d_ff, r] and
    factor_b [r, d] fp32 on the device (None with alpha = inf).  Returns
    (out [1, d], active_idx [1, d_ff], n_active [1])."""
    if out is None:
        out = torch.empty_like(x)
    if active_idx is None:
        active_idx = torch.empty((1, w.d_ff), dtype=torch.int32, device=x.device)
    if n_active is None:
        n_active = torch.empty(1, dtype=torch.int32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(WS_DECODE, 1, w, x.device)
    rank = 0 if factor_a is None else int(factor_a.shape[1])
    pa = None if factor_a is None else _ptr(factor_a)
    pb = None if factor_b is None else _ptr(factor_b)
    st = lib().sffn_decode_predicted(_ptr(x), w.ref(), pa, pb, rank, float(alpha), _ptr(out), _ptr(active_idx),
                                     _ptr(n_active), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sffn_decode_predicted")
    return out, active_idx, n_active


def decode_tiered(x: torch.Tensor, w: Weights, score: int, keep_ratio: float, core=None, out=None,
                  active_idx=None, n_active=None, workspace=None, stream=None):
    """Keep-ratio decode with a core set (int32 device tensor of column
    indices, ascending; None: no core).  Returns (out, active_idx, n_active)."""
    B = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    if active_idx is None:
        active_idx = torch.empty((B, w.d_ff), dtype=torch.int32, device=x.device)
    if n_active is None:
        n_active = torch.empty(B, dtype=torch.int32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(WS_DECODE, B, w, x.device)
    nc = 0 if core is None else int(core.numel())
    st = lib().sffn_decode_tiered(_ptr(x), B, w.ref(), int(score), float(keep_ratio), _ptr(core), nc, _ptr(out),
                                  _ptr(active_idx), _ptr(n_active), _ptr(workspace), workspace.numel(),
                                  _stream(stream))
    _check(st, "sffn_decode_tiered")
    return out, active_idx, n_active


def tier_core_set(calib_scores: torch.Tensor, k: int, n_core: int, core=None, workspace=None, stream=None):
    """Core set of a keep-ratio tier from calibration scores [N, d_ff] (fp32,
    device): int32 [n_core], ascending."""
    N, F = calib_scores.shape
    if core is None:
        core = torch.empty(n_core, dtype=torch.int32, device=calib_scores.device)
    if workspace is None:
        nb = lib().sffn_tier_core_workspace_size(N, F)
        if nb == 0:
            raise SffnError(ERR_SHAPE, "sffn_tier_core_workspace_size")
        workspace = torch.empty(nb, dtype=torch.uint8, device=calib_scores.device)
    st = lib().sffn_tier_core_set(_ptr(calib_scores), N, F, int(k), int(n_core), _ptr(core), _ptr(workspace),
                                  workspace.numel(), _stream(stream))
    _check(st, "sffn_tier_core_set")
    return core


def moe_progressive_k(layer: int) -> int:
    return int(lib().sffn_moe_progressive_k(int(layer)))


def moe_route(logits: torch.Tensor, cap: int, mass: float = 0.5, buckets=(3, 4, 5, 6), kmax=None, k_out=None,
              experts=None, weights=None, stream=None):
    """Adaptive expert top-K: (K [T], experts [T, kmax] ascending then -1,
    weights [T, kmax])."""
    T, E = logits.shape
    kmax = cap if kmax is None else kmax
    dev = logits.device
    if k_out is None:
        k_out = torch.empty(T, dtype=torch.int32, device=dev)
    if experts is None:
        experts = torch.empty((T, kmax), dtype=torch.int32, device=dev)
    if weights is None:
        weights = torch.empty((T, kmax), dtype=torch.float32, device=dev)
    bk = (C.c_int32 * len(buckets))(*buckets)
    st = lib().sffn_moe_route(_ptr(logits), T, E, int(cap), float(mass), bk, len(buckets), int(kmax), _ptr(k_out),
                              _ptr(experts), _ptr(weights), _stream(stream))
    _check(st, "sffn_moe_route")
    return k_out, experts, weights


def moe_block_budget(y_attn: torch.Tensor, mass: float, min_ratio: float = 0.10, max_ratio: float = 0.50,
                     block: int = 128, token_idx=None, n_tokens=None, ranges=None, n_ranges=None, workspace=None,
                     stream=None):
    """Block token budget: (token_idx [L], n_tokens [1], ranges [nblocks, 2], n_ranges [1])."""
    L, d = y_attn.shape
    dev = y_attn.device
    nblocks = (L + block - 1) // block
    if token_idx is None:
        token_idx = torch.empty(L, dtype=torch.int32, device=dev)
    if n_tokens is None:
        n_tokens = torch.empty(1, dtype=torch.int32, device=dev)
    if ranges is None:
        ranges = torch.empty((nblocks, 2), dtype=torch.int32, device=dev)
    if n_ranges is None:
        n_ranges = torch.empty(1, dtype=torch.int32, device=dev)
    if workspace is None:
        nb = lib().sffn_moe_budget_workspace_size(L, d)
        if nb == 0:
            raise SffnError(ERR_SHAPE, "sffn_moe_budget_workspace_size")
        workspace = torch.empty(nb, dtype=torch.uint8, device=dev)
    st = lib().sffn_moe_block_budget(_ptr(y_attn), L, d, float(mass), float(min_ratio), float(max_ratio), int(block),
                                     _ptr(token_idx), _ptr(n_tokens), _ptr(ranges), _ptr(n_ranges), _ptr(workspace),
                                     workspace.numel(), _stream(stream))
    _check(st, "sffn_moe_block_budget")
    return token_idx, n_tokens, ranges, n_ranges


def decode_noalloc(x: torch.Tensor, w: Weights, mode: int, score: int = SCORE_GATE, param: float = 0.0,
                   out=None, active_idx=None, n_active=None, stream=None):
    """sffn_decode with the library's built-in scratch array instead of a
    caller workspace, for callers that cannot allocate device memory (limit:
    NOALLOC_SCRATCH_BYTES of workspace; calls must not overlap on the GPU)."""
    B = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    if active_idx is None:
        active_idx = torch.empty((B, w.d_ff), dtype=torch.int32, device=x.device)
    if n_active is None:
        n_active = torch.empty(B, dtype=torch.int32, device=x.device)
    st = lib().sffn_decode_noalloc(_ptr(x), B, w.ref(), int(mode), int(score), float(param), _ptr(out),
                                   _ptr(active_idx), _ptr(n_active), _stream(stream))
    _check(st, "sffn_decode_noalloc")
    return out, active_idx, n_active


def gate_scores(x: torch.Tensor, w: Weights, score: int = SCORE_GATE, scores=None, workspace=None, stream=None):
    B = x.shape[0]
    if scores is None:
        scores = torch.empty((B, w.d_ff), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = alloc_workspace(WS_DECODE, B, w, x.device)
    st = lib().sffn_gate_scores(_ptr(x), B, w.ref(), int(score), _ptr(scores), _ptr(workspace),
                                workspace.numel(), _stream(stream))
    _check(st, "sffn_gate_scores")
    return scores


def token_select(y_attn: torch.Tensor, mass_thresh: float, recent_n: int, min_keep: int,
                 sel_idx=None, n_sel=None, workspace=None, stream=None):
    L, d = y_attn.shape
    if sel_idx is None:
        sel_idx = torch.empty(L, dtype=torch.int32, device=y_attn.device)
    if n_sel is None:
        n_sel = torch.empty(1, dtype=torch.int32, device=y_attn.device)
    if workspace is None:
        workspace = alloc_workspace(WS_SELECT, L, None, y_attn.device)
    st = lib().sffn_token_select(_ptr(y_attn), L, d, float(mass_thresh), int(recent_n), int(min_keep),
                                 _ptr(sel_idx), _ptr(n_sel), _ptr(workspace), workspace.numel(),
                                 _stream(stream))
    _check(st, "sffn_token_select")
    return sel_idx, n_sel


def prefill(x: torch.Tensor, y_attn: torch.Tensor, w: Weights, sel_idx: torch.Tensor, n_sel: torch.Tensor,
            out=None, workspace=None, stream=None):
    L = x.shape[0]
    if out is None:
        out = torch.empty_like(x)
    if workspace is None:
        workspace = alloc_workspace(WS_PREFILL, L, w, x.device)
    st = lib().sffn_prefill(_ptr(x), _ptr(y_attn), L, w.ref(), _ptr(sel_idx), _ptr(n_sel), _ptr(out),
                            _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sffn_prefill")
    return out


def read_device_error(workspace: torch.Tensor, stream=None) -> int:
    code = C.c_int32(0)
    _check(lib().sffn_read_device_error(_ptr(workspace), C.byref(code), _stream(stream)),
           "sffn_read_device_error")
    return int(code.value)


def decode_noalloc_read_error(stream=None) -> int:
    """Device error word of decode_noalloc's built-in array (read and cleared)."""
    code = C.c_int32(0)
    _check(lib().sffn_decode_noalloc_read_error(C.byref(code), _stream(stream)), "sffn_decode_noalloc_read_error")
    return int(code.value)


def schedule_preset(preset) -> FFNSchedule:
    """One of the presets ("speed", "balanced", "quality", "dense" or its enum)."""
    s = FFNSchedule()
    p = _PRESET[preset] if isinstance(preset, str) else int(preset)
    _check(lib().sffn_schedule_preset(p, C.byref(s)), "sffn_schedule_preset")
    return s


def schedule(dense_until: int, mass_thresh: float, recent_n: int, min_keep: int = 1,
             deep_layer_start: int = 2**31 - 1, mass_thresh_deep: float | None = None) -> FFNSchedule:
    return FFNSchedule(int(dense_until), int(deep_layer_start), float(mass_thresh),
                       float(mass_thresh if mass_thresh_deep is None else mass_thresh_deep), int(recent_n),
                       int(min_keep))


def schedule_mass(s: FFNSchedule, layer: int) -> float:
    return float(lib().sffn_schedule_mass(C.byref(s), int(layer)))


def prefill_layers(x: torch.Tensor, y_attn: list, weights: list, s: FFNSchedule, first_layer: int = 0,
                   out=None, sel_idx=None, n_sel=None, workspace=None, stream=None):
    """A stack of token-selective prefill layers; returns (out, sel_idx [n, L], n_sel [n])."""
    L = x.shape[0]
    n = len(weights)
    if out is None:
        out = torch.empty_like(x)
    if sel_idx is None:
        sel_idx = torch.empty((n, L), dtype=torch.int32, device=x.device)
    if n_sel is None:
        n_sel = torch.empty(n, dtype=torch.int32, device=x.device)
    if workspace is None:
        nb = max(int(lib().sffn_prefill_layers_workspace_size(L, w.ref())) for w in weights)
        if nb == 0:
            raise SffnError(ERR_SHAPE, "sffn_prefill_layers_workspace_size")
        workspace = torch.zeros(nb, dtype=torch.uint8, device=x.device)
    ya = (C.c_void_p * n)(*[_ptr(t) for t in y_attn])
    ws = (FFNWeights * n)(*[w.c for w in weights])
    st = lib().sffn_prefill_layers(_ptr(x), ya, L, n, ws, C.byref(s), int(first_layer), _ptr(out), _ptr(sel_idx),
                                   _ptr(n_sel), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sffn_prefill_layers")
    return out, sel_idx, n_sel
