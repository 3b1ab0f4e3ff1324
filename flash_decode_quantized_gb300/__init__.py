"""Fused dequant-on-load flash-decode over a resident, paged, block-quantized KV cache.

The compute lives in libkvq.so (CUDA, sm_103a) behind the C ABI in include/kvq.h; the
Python entry points in ``flash_decode_quantized_gb300.kvq`` carry the same names and only
marshal arguments.  Build the library with ``python -m flash_decode_quantized_gb300.build``.
"""

import importlib

__all__ = ["kvq", "build"]


def __getattr__(name):
    # Lazy: importing the package must not require the built library (the build step
    # imports it); importing `kvq` without the library raises ImportError.
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
