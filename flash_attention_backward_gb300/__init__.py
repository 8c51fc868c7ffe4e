"""GB300 (sm_103a) flash-attention backward over a raw F32/F16/q8_0/q4_0 K/V cache.

The computation lives in libfa_back.so (hand-written CUDA, C ABI in include/fa_back.h).
This package only marshals arguments: ``_native`` mirrors the C entry points under the same
names, and ``backward`` allocates outputs and workspace with PyTorch and calls ``fa_back``
on the current stream.
"""
from ._native import (  # noqa: F401
    FA_F16, FA_F32, FA_MASK_BITS, FA_MASK_F16, FA_Q4_0, FA_Q8_0, STATUS, NativeLibraryMissing, LIB_PATH,
    fa_back, fa_back_batched, fa_back_ext, fa_back_get_error, fa_back_noalloc, fa_back_nocopy, fa_back_plan_info,
    fa_back_profile, fa_back_workspace_size_nocopy,
    fa_back_profile_read, fa_back_selftest_timeout, fa_back_status_string, fa_back_strided,
    fa_back_strided_workspace_size, fa_back_test_wait_limit, fa_strides,
    fa_back_with_stats, fa_back_workspace_size, fa_back_workspace_size_min, fa_forward, fa_forward_workspace_size,
    fa_row_bytes, lib,
)
from .api import FaBackError, Workspace, backward, backward_strided, forward  # noqa: F401
