"""GB300-native (sm_103a) fused attention forward: prefill and Split-KV decode.

The computation lives in the CUDA library ``libfa_gb300.so`` (C ABI in
``include/fa.h``); this package only marshals arguments to it.
"""
from .fa import (  # noqa: F401
    FaError,
    fa_abi_version,
    fa_decode,
    fa_decode_plan,
    fa_decode_workspace_size,
    fa_forward,
    fa_forward_workspace_size,
    fa_selftest_wait_timeout,
    fa_status_string,
    fa_workspace_status,
)
