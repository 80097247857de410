"""KDA forward prefill for GB300 (sm_103a): a C-ABI CUDA library and its thin binding.

The compute lives in ``csrc/`` (hand-written CUDA for sm_103a) behind the C ABI
declared in ``include/kda.h``; :mod:`chunked_kda_delta_gb300.kda` marshals torch
tensors into that ABI through ctypes.  There is no CPU fallback: every entry
point raises if the compiled library is missing.
"""
from .kda import (  # noqa: F401
    KdaError,
    kda_prefill,
    kda_prefill_host,
    kda_status_string,
    kda_get_device_status,
    kda_release_workspaces,
    kda_workspace_bytes,
    kda_plan,
    kda_plan_varlen,
    kda_decode,
    STATE_F32,
    STATE_BF16,
    load_library,
    MODE_SERIAL,
    MODE_SEGMENT,
    MODE_AUTO,
)
