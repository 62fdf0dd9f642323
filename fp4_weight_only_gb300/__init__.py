"""GB300-native BF16-activation x FP4-weight (NVFP4 / MXFP4) GEMM.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/petit.h``); ``binding`` is its thin ctypes binding and ``synth``
draws seeded synthetic inputs.
"""

from . import synth  # noqa: F401

__all__ = ["binding", "synth", "build"]
