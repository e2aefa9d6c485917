"""GB300 (sm_103a) block-skipping causal prefill attention.

``bsa`` is the ctypes binding of the C library ``libbsa.so`` (include/bsa.h);
``build`` compiles it in-tree; ``api`` wraps the binding with torch tensors.
"""
from . import build, bsa  # noqa: F401
