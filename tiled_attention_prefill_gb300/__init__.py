"""Fused, tiled self-attention forward (prefill) for NVIDIA GB300 (sm_103a).

``forward`` and the other entry points live in :mod:`.fa` (a thin ctypes
binding over the C-ABI library ``libfa_gb300.so``); importing this package
does not load the library.
"""

import importlib

__version__ = "0.1.0"


def __getattr__(name):
    if name in ("forward", "load_library", "FAError", "check_device_status"):
        return getattr(importlib.import_module(__name__ + ".fa"), name)
    raise AttributeError(name)
