"""GB300-native activation-sparse gated FFN (decode GEMV + token-selective prefill).

The compute path is the C-ABI library ``libsffn.so`` (hand-written sm_103a CUDA
kernels, declared in ``include/sffn.h``); ``activation_sparse_ffn_gemv_gb300.sffn``
is the thin ctypes binding over it and loads the library on first use, raising
if it has not been built.  ``workloads`` holds the seeded synthetic inputs.
"""

__all__ = ["sffn", "workloads"]


def __getattr__(name):
    if name in ("sffn", "workloads"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
