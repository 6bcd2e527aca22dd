"""GB300-native (sm_103a) fused attention forward: prefill and Split-KV decode.

The computation lives in the CUDA library ``libfa_gb300.so`` (C ABI in
``include/fa.h``); this package only marshals arguments to it.
"""
from .fa import (  # noqa: F401
    FaError,
    fa_abi_version,
    fa_decode,
    fa_decode_masked,
    fa_decode_noalloc,
    fa_decode_noalloc_status,
    fa_decode_paged,
    fa_decode_plan,
    fa_decode_workspace_size,
    fa_forward,
    fa_forward_varlen,
    fa_forward_varlen_ex,
    fa_forward_varlen_window,
    fa_forward_varlen_workspace_size,
    fa_forward_paged,
    fa_forward_window,
    fa_forward_workspace_size,
    fa_kernel_launch_count,
    fa_selftest_wait_timeout,
    fa_set_main_kernel_events,
    fa_set_wait_timeout_ns,
    fa_status_string,
    fa_workspace_status,
)
