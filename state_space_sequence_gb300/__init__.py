"""GB300-native diagonal linear recurrence (DLR / diagonal SSM / S5) library.

The compute path is the C-ABI shared library ``libdlr.so`` (hand-written sm_103a CUDA
kernels, declared in ``include/dlr.h``); :mod:`state_space_sequence_gb300.dlr` is a thin
ctypes binding over it and :mod:`state_space_sequence_gb300.inputs` makes seeded inputs.
"""
__all__ = ["inputs"]
