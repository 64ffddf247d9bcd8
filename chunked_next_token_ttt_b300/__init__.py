"""libttt: chunked next-token test-time training on one B300 (sm_103a).

The compute path is the CUDA library libttt.so (built in-tree by
`python -m chunked_next_token_ttt_b300.build`); `Handle` is a thin ctypes
binding over its C ABI (include/ttt.h).
"""
from .ttt import Handle, TTTError, kernel_classes, load_library  # noqa: F401

__all__ = ["Handle", "TTTError", "kernel_classes", "load_library"]
