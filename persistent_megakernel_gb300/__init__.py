"""GB300-native batch-1 decode step as a persistent megakernel.

The CUDA path lives in ``csrc/`` behind the C ABI declared in ``include/dec.h``;
``binding`` is the thin ctypes layer over it. Importing the binding fails loudly
when the shared library has not been built: there is no CPU fallback.
"""
