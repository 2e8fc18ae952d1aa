"""GB300-native end-of-prefill KV-cache scoring, selection and compaction.

The compute path is libkvsel.so (CUDA for sm_103a, C ABI in include/kvsel.h);
``binding`` is its ctypes binding and ``datagen`` the seeded synthetic inputs.
Importing the package does not load the library; the first binding call does, and
raises if it is missing.
"""
from . import datagen  # noqa: F401

__all__ = ["datagen", "binding"]
