"""GB300-native block-sparse attention forward (FlexAttention-style).

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``, declared in ``include/fa.h``); ``fa.py`` is a thin ctypes
binding over it.  ``synth`` draws the seeded synthetic inputs.
"""
__all__ = ["fa", "synth"]
