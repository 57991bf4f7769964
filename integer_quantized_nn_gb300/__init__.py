"""GB300 (sm_103a) linear-quantized GEMM and implicit-GEMM convolution.

The compute path is the CUDA library libqnn.so (C ABI, include/qnn.h); the
``qnn`` module is its thin Python binding.  ``workloads`` holds the seeded
synthetic inputs of the benchmarked layer shapes.
"""
from . import qnn  # noqa: F401
from .qnn import *  # noqa: F401,F403
