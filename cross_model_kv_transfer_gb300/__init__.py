"""GB300-native cross-model KV-cache transfer (``kvx``).

The CUDA library (``libkvx.so``, C ABI declared in ``include/kvx.h``) does
the whole transfer; ``cross_model_kv_transfer_gb300.kvx`` is its thin ctypes
binding.  Submodules are imported on first use so that the seeded input
generators (``workloads``) can be used without loading the library.
"""
import importlib

__all__ = ["kvx", "workloads", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
