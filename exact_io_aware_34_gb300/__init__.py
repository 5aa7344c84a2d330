"""Exact, IO-aware attention forward pass (FlashAttention) for GB300 / sm_103a.

The computation runs in the CUDA library ``libfa.so`` (C ABI in include/fa.h);
this package holds its Python binding, its build step and the seeded input
generator.
"""
from .fa import (  # noqa: F401
    FA_ERR_CUDA,
    FA_ERR_INVALID_ARG,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_OK,
    FaError,
    fa_fwd,
    fa_fwd_fault_test,
    fa_get_device_status,
    fa_last_cuda_error,
    fa_naive_fwd,
    fa_naive_workspace_bytes,
    fa_status_string,
    load_library,
)
