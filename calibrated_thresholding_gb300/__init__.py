"""Top-theta attention on one GB300 (sm_103a).

The compute path is the C-ABI library ``libtopt.so`` (hand-written CUDA); the
Python layer in :mod:`calibrated_thresholding_gb300.topt` only marshals
arguments.  The library is loaded on first use and a missing build is an
error, never a fallback.
"""
