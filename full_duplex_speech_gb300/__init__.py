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
from . import _binding
from ._binding import *  # noqa: F401,F403  (the C ABI's names, one for one)

__all__ = [n for n in vars(_binding) if n.startswith("mamba2_")] + [
    "M2Error", "M2Dims", "M2RowNorm", "M2Lm", "M2LmLayer", "BF16", "F32", "NORM_NONE", "NORM_RMS", "NORM_GATED",
    "library_path", "load", "dims", "row_norm", "lm_model"]
