"""pooling_sliding_window_gb300 -- fused 2-D sliding-window operators for GB300.

The operators live in the CUDA library libfusedwin (C ABI in include/fusedwin.h,
kernels in csrc/); ``fusedwin`` is its Python binding and ``synth`` the seeded
input generator.  The binding is imported lazily so that the generator can be
used on machines without the CUDA toolkit.
"""

__all__ = ["fusedwin", "synth", "build"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
