"""GB300 (sm_103a) block-skipping causal prefill attention.

``bsa`` is the ctypes binding of the C library ``libbsa.so`` (include/bsa.h):
argument marshalling only, torch tensors passed by their device pointers;
``build`` compiles the library in-tree.
"""
from . import build, bsa  # noqa: F401
