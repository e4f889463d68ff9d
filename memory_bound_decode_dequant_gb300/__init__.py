"""GB300 decode step with fused dequantisation.

A thin ctypes binding over libmie.so (see include/mie.h).  Every function here only
marshals arguments -- device pointers of torch CUDA tensors, sizes, the current
stream -- and calls the library; all arithmetic of the decode step runs in the
library's CUDA kernels.  There is no CPU fallback: importing the binding without a
built libmie.so raises.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import __all__  # noqa: F401
