"""IQ4_XS x Q8_1 batched matmul for GB300 (sm_103a).

The computation runs in ``libiq4xs.so`` (hand-written CUDA kernels behind the
C ABI in ``include/iq4xs.h``); ``binding`` is a thin ctypes layer over it and
``synth`` generates seeded synthetic inputs.  Importing this package does not
load the CUDA library; the first call through ``binding`` does.
"""
from . import synth  # noqa: F401

__all__ = ["binding", "build", "synth"]
