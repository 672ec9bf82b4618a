"""GB300-native activation-sparse gated FFN (TwELL) library.

The compute path is the C-ABI CUDA library ``libtwell.so`` (built in-tree from
``csrc/``); ``twell`` is its thin ctypes binding and ``synthetic`` draws the
seeded inputs.  Importing ``twell`` fails loudly if the library is missing.
"""
__all__ = ["synthetic"]
