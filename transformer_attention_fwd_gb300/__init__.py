"""GB300-native scaled dot-product attention forward.

``attn`` (the ctypes binding over ``libattn.so``) is imported lazily so that
``inputs`` can be used on machines without the built library.
"""
from __future__ import annotations

import importlib

__all__ = ["attn", "inputs", "build"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
