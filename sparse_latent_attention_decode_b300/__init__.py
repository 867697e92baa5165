"""B300 (sm_103a) library for one decode step of absorbed, top-k-sparse latent
attention (DeepSeek-V3.2-Exp sparse MLA).

The compute lives in the CUDA shared library built from ``csrc/``; ``mla``
is the thin ctypes binding over its C ABI.  ``synth`` draws seeded inputs.
The binding is imported lazily so that input generation works on machines
without the built library.
"""

__all__ = ["mla", "synth"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
