"""Low-bit (INT4/INT2) KV-cache decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libkvq.so`` built from ``csrc/``; this
package holds its thin ctypes binding (``kvq``), a cache allocator over torch
device memory (``kvq.KVCache``), the build step (``_build``) and the seeded
input generator (``synth``).  Importing the package loads nothing; the library
is loaded on first use, and an absent or unbuilt library raises instead of
falling back to anything else.
"""

import importlib

__all__ = ["kvq", "synth"]


def __getattr__(name):
    if name in ("kvq", "synth", "_build"):
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
