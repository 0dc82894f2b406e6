"""GB300 (sm_103a) Mamba2 mixer core of the Nemotron-H language model in
NemotronLabs VoiceChat: causal conv1d + SiLU over x|B|C, softplus dt, and the
selective state-space recurrence, as a chunked (SSD) scan for full-history
recompute / prefill and as a single-frame cached step for many sessions; and
around it the gated output norm, the 4-bit projections and the cached decode
of the model's grouped-query attention layers.

Every step of the computation runs in the CUDA kernels of libmamba2.so
(C ABI: include/mamba2.h). This package only marshals arguments: torch
tensors (or raw device pointers) in, status codes checked, nothing computed
in Python. Importing it loads the library; a missing library is an error,
never a silent fallback.
"""
from ._binding import (  # noqa: F401
    M2Error,
    M2Dims,
    BF16,
    F32,
    library_path,
    load,
    dims,
    mamba2_scan_workspace_bytes,
    mamba2_conv_scan,
    mamba2_conv_scan_varlen,
    mamba2_scan_prepare_bc,
    mamba2_scan_chunks,
    mamba2_step_workspace_bytes,
    mamba2_gated_norm,
    mamba2_qlinear,
    mamba2_attn_decode,
    mamba2_attn_decode_workspace_bytes,
    mamba2_step,
    mamba2_step_noalloc,
    mamba2_step_noalloc_max_bytes,
    mamba2_status_string,
    mamba2_last_cuda_error,
    mamba2_device_error,
)

__all__ = [
    "M2Error", "M2Dims", "BF16", "F32", "library_path", "load", "dims",
    "mamba2_scan_workspace_bytes", "mamba2_conv_scan", "mamba2_conv_scan_varlen", "mamba2_scan_prepare_bc", "mamba2_scan_chunks", "mamba2_step_workspace_bytes", "mamba2_gated_norm", "mamba2_qlinear",
    "mamba2_attn_decode", "mamba2_attn_decode_workspace_bytes",
    "mamba2_step", "mamba2_step_noalloc", "mamba2_step_noalloc_max_bytes", "mamba2_status_string", "mamba2_last_cuda_error", "mamba2_device_error",
]
