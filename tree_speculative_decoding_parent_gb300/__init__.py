"""GB300-native (sm_103a) verify-and-graft step of tree speculative decoding.

The compute lives in libgt.so (CUDA kernels behind the C ABI of include/gt.h), built
in-tree by ``build.build()``; ``gt`` is its ctypes binding and ``step`` runs one whole
step through it.
"""
from . import build, gt  # noqa: F401
