"""GB300 (sm_103a) fused exact attention: the forward (16-bit, grouped K/V
heads, 8-bit inputs), its backward, and decoding over a paged K/V cache.

The compute lives in ``libfa.so`` (CUDA, built by ``build.build()``); the
Python layer in ``fa.py`` only marshals arguments into its C ABI
(``include/fa.h``).  Submodules are imported lazily so that the input
generator can be used without the library.
"""
__all__ = ["fa", "build", "inputs", "metrics"]


def __getattr__(name):
    import importlib
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
