"""MLA attention computed from the compressed latent, on GB300 (sm_103a).

The compute lives in ``libmla.so`` (hand-written CUDA behind a C ABI, declared in
``include/mla.h``); :mod:`.mla` is the thin ctypes binding with the same entry-point
names.  The binding loads the library on first use and raises if it is missing:
there is no other implementation behind it.
"""
from . import configs, inputs, mla  # noqa: F401

__all__ = ["configs", "inputs", "mla"]
