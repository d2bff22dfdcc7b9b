"""Exact scaled-dot-product attention for GB300 (sm_103a): C-ABI library + binding.

``forward``/``backward`` take torch CUDA tensors; ``fa_*`` are the raw C-ABI
calls with the names of include/fa.h.  The library is loaded on first use.
"""
from .fa import (FaError, backward, fa_bwd, fa_bwd_workspace_bytes, fa_device_status,  # noqa: F401
                 fa_fwd, fa_status_string, forward, load)
