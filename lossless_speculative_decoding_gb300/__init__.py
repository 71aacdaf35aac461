"""GB300-native greedy, lossless speculative-decoding verify step.

The compute path is the CUDA library ``libspec.so`` (sources in ``csrc/``,
C ABI in ``include/spec.h``); ``binding`` marshals arguments to it through
ctypes and ``runtime`` adds a small object wrapper. Build the library with
``build.build()``.
"""
from . import binding  # noqa: F401

__all__ = ["binding"]
