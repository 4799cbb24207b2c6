"""QSA sparse-attention decode step on one GB300 (sm_103a).

The compute runs in the hand-written CUDA library libqsa_gb300.so through the
C ABI of include/qsa.h; this package is its thin Python binding.  Importing
the package does not load the library; the first call does, and it raises if
the library has not been built.
"""
from ._native import (ERR_BAD_BLOCK, ERR_BAD_SLOT, ERR_CAPACITY, ERR_CUDA, ERR_INVALID_ARG,  # noqa: F401
                      ERR_NO_DEVICE, ERR_OUT_OF_SLOTS, ERR_STALE_HANDLE, ERR_TIMEOUT, KV_HBM,
                      KV_BF16, KV_FP8, KV_HOST, KV_HOST_RING, OK, Handle, QsaError, lib)
from .api import Cache  # noqa: F401
