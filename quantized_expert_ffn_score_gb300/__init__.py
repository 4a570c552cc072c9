"""GB300 (sm_103a) MoE-layer forward: router/top-k, bucketing, MXFP4 and RVQ3
expert FFNs decoded inside hand-written CUDA kernels, and the gate-weighted
combine, behind the C ABI in include/moe.h (libmoe_gb300.so).

`moe` is the ctypes binding (same names as the C entry points); `build` compiles
the library in-tree; `synthetic` materialises seeded layers in HBM.
"""
from . import build  # noqa: F401

__all__ = ["build", "moe", "synthetic"]


def __getattr__(name):
    if name in ("moe", "synthetic"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
