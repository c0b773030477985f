"""GB300-native quantized-weight matvec: CQ (codebook + FWHT) and F8 E4M3/E8M0.

The compute path is the C-ABI library ``libqmv.so`` (hand-written CUDA for
sm_103a, declared in ``include/qmv.h``); ``qmv`` is its thin ctypes binding.
Importing this package does not load the library; ``qmv`` does, and fails
loudly when it is missing.
"""
__all__ = ["synth", "qmv"]
