"""GB300-native fused attention (sm_103a): forward and backward, exported through
libattn's C ABI.

The Python layer only marshals arguments: every step of both passes runs
in the CUDA kernels of ``libattn.so``.  Importing this package does not load
the library; the first call does, and it raises if the library is missing.
"""
from ._binding import (  # noqa: F401
    ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT,
    ATTN_DTYPE_BF16, ATTN_DTYPE_F16, AttnError, attn_fwd, attn_fwd_ptr, attn_fwd_ex_ptr, attn_fwd_splitkv, attn_fwd_splitkv_ptr,
    attn_fwd_splitkv_workspace_size, attn_fwd_splitkv_noalloc_ptr, attn_status_str,
    attn_last_device_status, attn_check_device_status,
    attn_kernel_launches, attn_debug_wait_timeout, attn_debug_unit_rates, attn_debug_unit_schedule, library_path,
    load_library,
    exported_symbols, attn_bwd, attn_bwd_ptr, attn_bwd_workspace_size,
)
