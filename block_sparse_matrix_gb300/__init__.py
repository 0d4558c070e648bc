"""Block-sparse matrix multiplication for GB300 (sm_103a).

``bsmm`` is the ctypes binding of the CUDA library ``libbsmm.so`` (C ABI in
include/bsmm.h); ``workloads`` holds the seeded synthetic inputs.
"""
from .bsmm import BlocksparseMatMul, BsmmError, group_param_grads  # noqa: F401
