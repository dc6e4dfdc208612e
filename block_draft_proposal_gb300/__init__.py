"""GB300-native DFlash2 draft-proposal hot path.

The compute lives in ``libdflash2.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/dflash2.h``).  :mod:`.dflash2` is the thin ctypes
binding; :mod:`.synth` draws seeded synthetic inputs.  Importing this package
loads nothing: the binding opens the library on first use and raises if it is
missing.
"""
__all__ = ["dflash2", "synth"]
