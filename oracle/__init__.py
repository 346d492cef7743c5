"""fp64 CPU oracle for the activation-sparse gated FFN -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its binding)
never does, and this package imports nothing from it.

The arithmetic lives in ``sffn_oracle.c`` (plain C, fp64, ascending-index
loops); this module only compiles it with gcc and marshals numpy arrays.  Raw
input buffers are passed as stored (fp32, bf16 bit patterns as uint16, packed
int4 codes as uint8 with fp16 scale bits as uint16) and decoded exactly by the C
code.

Parity status: every function is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute force on tiny inputs, numpy fp64 special cases, printed
worked values from the pages); none is "parity unpinned".  The submodules
``predictor`` (low-rank gate predictor), ``tiers`` (keep-ratio tier tables with a
core set) and ``moe`` (adaptive expert top-K, block token budget) are pinned by
``tests/test_predictor_oracle.py``, ``tests/test_tiers_oracle.py`` and
``tests/test_moe_oracle.py``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sffn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Stored element formats (must match the enum in sffn_oracle.c).
F32, BF16, INT4_G64, F64 = 0, 1, 2, 3
RELU, SILU = 0, 1
EXACT, THRESHOLD, KEEP_RATIO = 0, 1, 2
SCORE_GATE, SCORE_GATE_UP = 0, 1


def build(force: bool = False) -> str:
    """Compile sffn_oracle.c into _build/liboracle.so (plain -O2, no fast-math)."""
    with _lock:
        os.makedirs(_BUILD, exist_ok=True)
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


class _Mat(C.Structure):
    _fields_ = [("fmt", C.c_int), ("rows", C.c_int), ("cols", C.c_int),
                ("data", C.c_void_p), ("scales", C.c_void_p)]


class _FFN(C.Structure):
    _fields_ = [("d_model", C.c_int), ("d_ff", C.c_int), ("act", C.c_int),
                ("w_gate", _Mat), ("w_up", _Mat), ("w_downT", _Mat),
                ("b_gate", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = C.CDLL(path)
        P = C.c_void_p
        L.orc_bf16_to_f64.argtypes = [C.c_uint16]
        L.orc_bf16_to_f64.restype = C.c_double
        L.orc_f16_to_f64.argtypes = [C.c_uint16]
        L.orc_f16_to_f64.restype = C.c_double
        L.orc_f64_to_bf16_rne.argtypes = [C.c_double]
        L.orc_f64_to_bf16_rne.restype = C.c_uint16
        L.orc_mat_to_f64.argtypes = [C.POINTER(_Mat), P]
        L.orc_mat_to_f64.restype = None
        L.orc_act.argtypes = [C.c_int, C.c_double]
        L.orc_act.restype = C.c_double
        L.orc_down_norms.argtypes = [C.POINTER(_FFN), P]
        L.orc_down_norms.restype = None
        L.orc_keep_count.argtypes = [C.c_int, C.c_double]
        L.orc_keep_count.restype = C.c_int
        L.orc_row_bytes.argtypes = [C.c_int, C.c_int]
        L.orc_row_bytes.restype = C.c_double
        L.orc_bytes_kept.argtypes = [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]
        L.orc_bytes_kept.restype = C.c_double
        L.orc_decode.argtypes = [C.POINTER(_FFN), C.POINTER(_Mat), C.c_int, C.c_int, C.c_int,
                                 C.c_double, P, P, P, P, P, P, P, P, P, P, P, P, C.c_int]
        L.orc_decode.restype = C.c_int
        L.orc_token_norms.argtypes = [C.POINTER(_Mat), P]
        L.orc_token_norms.restype = None
        L.orc_mass_select.argtypes = [C.c_int, P, C.c_double, C.c_int, C.c_int, P, P, P, P]
        L.orc_mass_select.restype = C.c_int
        L.orc_residual.argtypes = [C.POINTER(_Mat), C.POINTER(_Mat), P]
        L.orc_residual.restype = None
        L.orc_prefill_rows.argtypes = [C.POINTER(_FFN), C.POINTER(_Mat), C.POINTER(_Mat), P, P,
                                       C.c_int, P, P, C.c_int]
        L.orc_prefill_rows.restype = C.c_int
        _lib = L
    return _lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _np(a):
    """Accept numpy arrays or CPU torch tensors (bf16 is viewed as uint16 bits)."""
    if a is None:
        return None
    if not isinstance(a, np.ndarray):
        import torch  # only for tensor -> numpy views
        t = a.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16 or t.dtype == torch.float16:
            t = t.view(torch.int16)
            return t.numpy().view(np.uint16)
        return t.numpy()
    return np.ascontiguousarray(a)


class Mat:
    """A stored matrix: fmt in {F32, BF16, INT4_G64, F64}; keeps buffers alive."""

    def __init__(self, fmt, data, rows, cols, scales=None):
        self.fmt, self.rows, self.cols = fmt, int(rows), int(cols)
        self.data = _np(data)
        self.scales = _np(scales)
        want = {F32: np.float32, BF16: np.uint16, INT4_G64: np.uint8, F64: np.float64}[fmt]
        if self.data.dtype != want:
            self.data = self.data.astype(want) if fmt in (F32, F64) else self.data.view(want)
        n = self.rows * self.cols
        if fmt == INT4_G64:
            assert self.data.size == n // 2 and self.cols % 64 == 0
            if self.scales.dtype != np.uint16:
                self.scales = self.scales.view(np.uint16)
            assert self.scales.size == self.rows * (self.cols // 64)
        else:
            assert self.data.size == n, (self.data.size, n)
        self.c = _Mat(fmt, self.rows, self.cols, _ptr(self.data), _ptr(self.scales))

    def to_f64(self):
        out = np.empty((self.rows, self.cols), np.float64)
        lib().orc_mat_to_f64(C.byref(self.c), _ptr(out))
        return out


class FFN:
    """One FFN layer: w_gate, w_up, w_downT are Mat [F, d]; b_gate float32 [F] or None."""

    def __init__(self, w_gate: Mat, w_up: Mat, w_downT: Mat, act: int, b_gate=None):
        self.w_gate, self.w_up, self.w_downT = w_gate, w_up, w_downT
        self.d_ff, self.d_model = w_gate.rows, w_gate.cols
        self.act = act
        self.b_gate = None if b_gate is None else np.ascontiguousarray(_np(b_gate), np.float32)
        self.c = _FFN(self.d_model, self.d_ff, act, w_gate.c, w_up.c, w_downT.c, _ptr(self.b_gate))


def bf16_to_f64(bits: int) -> float:
    return lib().orc_bf16_to_f64(int(bits))


def f16_to_f64(bits: int) -> float:
    return lib().orc_f16_to_f64(int(bits))


def f64_to_bf16_bits(v: float) -> int:
    return int(lib().orc_f64_to_bf16_rne(float(v)))


def act(kind: int, z: float) -> float:
    return lib().orc_act(int(kind), float(z))


def keep_count(F: int, keep_ratio: float) -> int:
    return lib().orc_keep_count(int(F), float(keep_ratio))


def row_bytes(fmt: int, d: int) -> float:
    return lib().orc_row_bytes(int(fmt), int(d))


def bytes_kept(fmt: int, d: int, F: int, score_kind: int, n_active: int) -> float:
    return lib().orc_bytes_kept(int(fmt), int(d), int(F), int(score_kind), int(n_active))


def down_norms(ffn: FFN) -> np.ndarray:
    out = np.empty(ffn.d_ff, np.float64)
    lib().orc_down_norms(C.byref(ffn.c), _ptr(out))
    return out


def decode(ffn: FFN, x: Mat, mode: int, score_kind: int = SCORE_GATE, param: float = 0.0,
           given_idx=None, given_n=None, nthreads: int = 1, details: bool = False):
    """Decode x [B, d] through one layer.  Returns a dict with ``out`` [B, d]
    fp64, ``active_idx`` [B, F] (valid up to ``n_active[b]``), ``n_active`` [B],
    and with ``details`` also g, a, u, score, cond [B, F], cut [B], norms [F].
    When ``given_idx``/``given_n`` are supplied, ``out`` is computed on that
    set (the oracle's own selection is still returned)."""
    B, F, d = x.rows, ffn.d_ff, ffn.d_model
    out = np.zeros((B, d), np.float64)
    idx = np.zeros((B, F), np.int32)
    n = np.zeros(B, np.int32)
    det = {k: np.zeros((B, F), np.float64) for k in ("g", "a", "u", "score", "cond")} if details else {}
    cut = np.zeros(B, np.float64) if details else None
    norms = np.zeros(F, np.float64) if details else None
    gi = None if given_idx is None else np.ascontiguousarray(given_idx, np.int32)
    gn = None if given_n is None else np.ascontiguousarray(given_n, np.int32)
    if gi is not None:
        assert gi.shape == (B, F) and gn.shape == (B,)
    rc = lib().orc_decode(C.byref(ffn.c), C.byref(x.c), B, mode, score_kind, float(param),
                          _ptr(gi), _ptr(gn), _ptr(out), _ptr(idx), _ptr(n),
                          _ptr(det.get("g")), _ptr(det.get("a")), _ptr(det.get("u")),
                          _ptr(det.get("score")), _ptr(det.get("cond")), _ptr(cut), _ptr(norms),
                          int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode: bad argument")
    res = {"out": out, "active_idx": idx, "n_active": n}
    if details:
        res.update(det)
        res["cut"], res["norms"] = cut, norms
    return res


def token_norms(y_attn: Mat) -> np.ndarray:
    s = np.empty(y_attn.rows, np.float64)
    lib().orc_token_norms(C.byref(y_attn.c), _ptr(s))
    return s


def mass_select(s, mass_thresh: float, recent_n: int, min_keep: int):
    """Returns (sel_idx ascending, prefix_idx in selection order)."""
    s = np.ascontiguousarray(s, np.float64)
    L = s.size
    sel = np.zeros(max(L, 1), np.int32)
    pre = np.zeros(max(L, 1), np.int32)
    n = np.zeros(1, np.int32)
    k = np.zeros(1, np.int32)
    rc = lib().orc_mass_select(L, _ptr(s), float(mass_thresh), int(recent_n), int(min_keep),
                               _ptr(sel), _ptr(n), _ptr(k), _ptr(pre))
    if rc < 0:
        raise ValueError("oracle mass_select: bad argument")
    return sel[: n[0]].copy(), pre[: k[0]].copy()


def residual(X: Mat, Y_attn: Mat) -> np.ndarray:
    """bf16 bits of Y = bf16_rne(X + Y_attn), [L, d] uint16."""
    out = np.empty((X.rows, X.cols), np.uint16)
    lib().orc_residual(C.byref(X.c), C.byref(Y_attn.c), _ptr(out))
    return out


def prefill_rows(ffn: FFN, X: Mat, Y_attn: Mat, selected_mask, rows, nthreads: int = 1):
    """Returns (z [n, d] fp64, out bits [n, d] uint16) for the requested rows."""
    rows = np.ascontiguousarray(rows, np.int32)
    sel = np.ascontiguousarray(selected_mask, np.uint8)
    assert sel.size == X.rows
    z = np.zeros((rows.size, ffn.d_model), np.float64)
    out = np.zeros((rows.size, ffn.d_model), np.uint16)
    rc = lib().orc_prefill_rows(C.byref(ffn.c), C.byref(X.c), C.byref(Y_attn.c), _ptr(sel),
                                _ptr(rows), rows.size, _ptr(z), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle prefill: bad argument")
    return z, out
