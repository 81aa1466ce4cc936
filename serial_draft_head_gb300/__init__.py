"""GB300 (sm_103a) persistent serial Markov draft walk.

The CUDA library (``_build/libdspark_walk.so``) is the product; ``walk`` is a
thin ctypes binding of its C ABI (``include/dspark_walk.h``).
"""
from . import walk  # noqa: F401
from .walk import Walk, WalkError  # noqa: F401
