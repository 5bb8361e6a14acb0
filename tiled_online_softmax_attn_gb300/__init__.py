"""GB300 (sm_103a) exact attention forward, O = softmax(Q K^T * scale) V.

The work runs in hand-written CUDA kernels behind the C ABI of
``include/fa.h`` (``libfa_gb300.so``); this package is its thin Python
binding.  Build the library with ``tiled_online_softmax_attn_gb300.build.build()``.
"""
from ._binding import (FA_BF16, FA_ERR_CUDA, FA_ERR_INVALID_ARG, FA_ERR_TIMEOUT,  # noqa: F401
                       FA_ERR_UNSUPPORTED, FA_FLAG_GENERAL_PATH, FaParams, FA_FLAG_TEST_SKIP_KV_LOAD, FA_FP32, FA_OK, FAError,
                       attention_workspace_size, backward_plan, backward_workspace_size, check_device_error,
                       fa_attention, fa_backward, fa_forward,
                       forward_host, forward_raw,
                       host_workspace_size, last_error, last_status, load, plan, version, workspace_size)
