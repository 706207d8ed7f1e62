"""Layout-aware reduce-scatter math and all-gather placement for FSDP2-style
per-parameter storage on one GB300 (sm_103a).

The compute lives in libtide.so (CUDA kernels behind the C ABI declared in
include/tide.h); this package is its ctypes binding plus a small Layout
convenience wrapper.
"""
from .tide import *  # noqa: F401,F403
from .tide import PointerTable, TideError  # noqa: F401
from .layout import Layout  # noqa: F401
