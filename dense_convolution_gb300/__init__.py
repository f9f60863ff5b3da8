"""Forward 2-D convolution for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI shared library built from ``csrc/`` (declared
in ``include/conv2d.h``); ``capi`` binds it with ctypes and ``conv`` offers a
PyTorch-tensor convenience layer (PyTorch supplies device memory and the
stream only).  Importing this package loads nothing; the library is loaded on
first use and raises if it has not been built.
"""

__all__ = ["capi", "conv"]
