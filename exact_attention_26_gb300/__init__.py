"""Exact scaled-dot-product attention for GB300 (sm_103a): C-ABI library + binding.

``forward``/``backward``/``decode`` take torch CUDA tensors; ``fa_*`` are the raw C-ABI
calls with the names of include/fa.h.  The library is loaded on first use.
"""
from .fa import (FaError, backward, backward_varlen, decode, decode_paged, fa_bwd,  # noqa: F401
                 fa_bwd_workspace_bytes, fa_decode, fa_decode_num_splits, fa_decode_paged,
                 fa_decode_uses_tensor_cores,
                 fa_decode_paged_num_splits, fa_decode_paged_workspace_bytes,
                 fa_decode_workspace_bytes, fa_device_status, fa_fwd, fa_fwd_fp8, fa_fwd_varlen,
                 fa_fwd_split_segments, fa_fwd_workspace_bytes, fa_fwd_ws, fwd_split_segments,
                 fa_probe_read_bandwidth, fa_probe_unit_rates, fa_quantize_fp8,
                 fa_quantize_fp8_workspace_bytes, fa_status_string, forward, forward_fp8,
                 forward_varlen, load, probe_read_bandwidth, probe_unit_rates, quantize_fp8)
from .fa import FA_ERR_INVALID_ARG, FA_ERR_MISALIGNED, FA_ERR_WORKSPACE, FA_OK  # noqa: F401
from .pipeline import HostPipeline  # noqa: F401,E402
