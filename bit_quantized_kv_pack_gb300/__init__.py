"""Low-bit (INT4/INT2) KV-cache decode attention for GB300 (sm_103a).

The compute path is the C-ABI library ``libkvq.so`` built from ``csrc/``; this
package holds its thin ctypes binding (``kvq``), a cache allocator over torch
device memory (``KVCache``) and the seeded input generator (``synth``).
Importing the package loads nothing; the library is loaded on first use and an
absent or unbuilt library raises instead of falling back to anything else.
"""

__all__ = ["kvq", "synth", "build"]


def __getattr__(name):
    if name == "kvq":
        from . import kvq as _kvq
        return _kvq
    if name == "synth":
        from . import synth as _synth
        return _synth
    if name == "build":
        from ._build import build as _b
        return _b
    raise AttributeError(name)
