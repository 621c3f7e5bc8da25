"""GB300-native scaled dot-product attention forward.

``attn`` (the ctypes binding over ``libattn.so``) is imported lazily so that
``inputs`` can be used on machines without the built library.
"""
from __future__ import annotations

__all__ = ["attn", "inputs"]


def __getattr__(name):
    if name == "attn":
        from . import attn as _attn
        return _attn
    if name == "inputs":
        from . import inputs as _inputs
        return _inputs
    raise AttributeError(name)
