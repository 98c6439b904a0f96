"""GB300-native per-token NVFP4 W4A4 linear-layer path.

The compute lives in a C-ABI shared library (nvfp4_precision_rl_gb300/_build/
libnvfp4.so, declared in include/nvfp4.h, hand-written CUDA for sm_103a).
`nvfp4_precision_rl_gb300.ops` is the thin ctypes binding with the same names;
it refuses to run when the library is not built (there is no CPU fallback).

Importing this package does not load the library; `ops` loads it on first use.
"""
import importlib

__all__ = ["ops", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
