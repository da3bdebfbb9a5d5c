"""Gated DeltaNet chunked forward pass on GB300 (sm_103a).

The compute path is libgdn.so (include/gdn.h); this package holds its thin
Python binding (``binding``), the build step (``build``) and the seeded
synthetic input recipes (``inputs``).  Submodules are imported lazily so that
``inputs`` can be used without loading the CUDA library.
"""
__all__ = ["binding", "build", "inputs"]


def __getattr__(name):
    import importlib
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
