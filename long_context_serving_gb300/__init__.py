"""Block-sparse decode attention for GB300 (sm_103a).

``bsattn`` is the thin ctypes binding of ``libbsattn.so`` (the C ABI declared in
``include/bsattn.h``); ``layer`` holds the device buffers of one attention layer;
``build`` compiles the library in-tree with nvcc.
"""
from . import bsattn  # noqa: F401  (loads nothing until the first call)
