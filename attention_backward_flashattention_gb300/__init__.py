"""GB300-native (sm_103a) fused attention forward/backward.

The compute path is the C-ABI library ``libattn_gb300.so`` built from
``csrc/`` (hand-written CUDA for sm_103a).  ``binding`` wraps its entry points
with the same names; nothing here computes attention on the CPU.
Submodules are imported on first use so that importing the package never
loads the CUDA library by itself.
"""
import importlib

__all__ = ["binding", "synthetic"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
