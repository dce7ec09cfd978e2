"""Paged sliding-window attention for Gemma-style hybrid decoders on GB300.

The compute lives in ``libpsw.so`` (hand-written CUDA for sm_103a behind a C
ABI, declared in ``include/psw.h``). ``paged_sliding_window_gb300.binding``
marshals torch tensors into that ABI; importing this package does not load
the library (``workloads`` is usable without a GPU).
"""

__all__ = ["binding", "workloads", "build"]


def __getattr__(name):
    if name in ("binding", "workloads", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
