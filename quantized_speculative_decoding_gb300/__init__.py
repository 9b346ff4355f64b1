"""GB300-native hot path of quantized speculative decoding.

The compute lives in ``libsd.so`` (CUDA kernels for sm_103a behind the C ABI
declared in ``include/sd.h``).  ``binding`` is a thin ctypes layer over that
ABI with the same function names; it raises if the library is missing rather
than falling back to anything else.  ``synth`` holds the seeded synthetic
input recipes.  Nothing is imported eagerly so that the input recipes can be
used on machines without the library.
"""
__all__ = ["binding", "synth"]
