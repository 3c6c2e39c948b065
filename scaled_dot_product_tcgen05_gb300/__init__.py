"""Fused scaled-dot-product attention forward for GB300 (sm_103a).

The compute path is one hand-written CUDA kernel (tcgen05 MMA, TMEM
accumulators, TMA-fed shared memory, online softmax) behind the C ABI of
include/attn.h; this package is a thin ctypes binding over it.
"""
from ._binding import (  # noqa: F401
    ATTN_ERR_BAD_SEQLENS,
    ATTN_ERR_CUDA,
    ATTN_ERR_DEVICE_TIMEOUT,
    ATTN_ERR_INVALID_ARG,
    ATTN_ERR_MISALIGNED,
    ATTN_ERR_UNSUPPORTED,
    ATTN_OK,
    EXPORTED,
    AttnError,
    attn_bwd,
    attn_check,
    attn_decode,
    attn_fwd,
    attn_fwd_fp8,
    attn_fwd_raw,
    attn_fwd_window_raw,
    attn_merge,
    bwd_workspace_bytes,
    decode_workspace_bytes,
    fp8_workspace_bytes,
    last_launch,
    load_library,
    num_sms,
    status_string,
)
