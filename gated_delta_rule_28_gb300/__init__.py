"""GB300 (sm_103a) chunked gated-delta-rule scan behind a C ABI (include/gdn.h).

``binding``   ctypes front end with the C entry-point names (marshalling only).
``api``       tensor-level calls that allocate with PyTorch and call the binding.
``workloads`` seeded synthetic inputs shaped like the pages' workloads.
``build``     in-tree nvcc build of libgdn.so for sm_103a.
"""
from . import binding  # noqa: F401
