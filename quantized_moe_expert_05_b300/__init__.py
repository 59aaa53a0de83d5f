"""B300-native batch-1 quantised MoE expert block.

``libfmoe.so`` (built from ``csrc/`` by ``build.py``) holds the CUDA kernels
behind the C ABI declared in ``include/fmoe.h``; ``fmoe`` is its ctypes
binding.  Importing the package does not load the library; importing
``quantized_moe_expert_05_b300.fmoe`` does, and fails if it is missing.
"""
import importlib

__all__ = ["build", "fmoe"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
