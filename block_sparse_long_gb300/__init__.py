"""CoSA block-sparse long-context prefill for GB300 (sm_103a).

The hot path lives in libcosa.so (CUDA kernels behind the C ABI of include/cosa.h);
``block_sparse_long_gb300.cosa`` is its thin Python binding.
"""
from .cosa import (COSA_OK, COSA_ERR_INVALID_ARG, COSA_ERR_UNSUPPORTED, COSA_ERR_CUDA, COSA_ERR_DEVICE_TIMEOUT,
                   COSA_ERR_WORKSPACE, COSA_ERR_BAD_INPUT, VISIT_COMPUTED, VISIT_SKIPPED, VISIT_IGNORED, EXPORTS,
                   CosaError, CosaParams, cosa_prefill_workspace_size, cosa_proxy_select, cosa_proxy_select_static,
                   cosa_proxy_workspace_size, cosa_sparse_prefill, cosa_status_string, cosa_version, library,
                   make_params, params_for, stage1_pitch)

__all__ = [n for n in dir() if n.startswith(("cosa_", "COSA_", "VISIT_")) or n in (
    "CosaError", "CosaParams", "EXPORTS", "library", "make_params", "params_for", "stage1_pitch")]
