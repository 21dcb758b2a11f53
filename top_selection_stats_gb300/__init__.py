"""GB300-native batched top-k / top-p truncation and sampling.

A thin binding over the C ABI in ``include/smp.h`` (``libsmp.so``, hand-written
sm_103a CUDA).  This module only marshals arguments: torch supplies device
memory and the current stream, every step of the computation runs in the CUDA
kernels.  There is no fallback: if the library is missing, calls raise.
"""
from .binding import (SMP_OK, SMP_ERR_EMPTY, SMP_ERR_NONFINITE, SMP_ERR_INVALID_PARAM,
                      SMP_ERR_TIMEOUT, SMP_ERR_CUDA, SMP_ERR_CAPACITY, PATH_NAMES, Sampler,
                      SmpError, lib_path, load_library, sample_noalloc)

__all__ = ["Sampler", "SmpError", "load_library", "lib_path", "sample_noalloc", "SMP_OK",
           "SMP_ERR_EMPTY", "SMP_ERR_NONFINITE", "SMP_ERR_INVALID_PARAM", "SMP_ERR_TIMEOUT", "SMP_ERR_CUDA",
           "SMP_ERR_CAPACITY", "PATH_NAMES"]
