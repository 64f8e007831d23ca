"""GB300-native Sparse State Expansion (SSE) layer: a C-ABI CUDA library
(``libsse``) for sm_103a plus a thin ctypes binding.

Submodules are imported lazily so that the synthetic-input module can be used
on machines without a GPU.
"""
import importlib

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
