"""NVFP4 fake-quantized attention training (Attn-QAT) for GB300 (sm_103a).

The compute lives in ``libnvfp4attn.so`` (C ABI: include/nvfp4attn.h, kernels in
``csrc/``).  ``api`` is the PyTorch binding, ``workloads`` the seeded synthetic
inputs.  Importing this package loads nothing; the library is loaded on the
first call and its absence raises ``NvqLibraryError``.
"""
from ._lib import NvqError, NvqLibraryError  # noqa: F401

__all__ = ["NvqError", "NvqLibraryError"]
