"""GB300-native grouped-query online-softmax attention.

The compute lives in ``libattn_gqa.so`` (CUDA kernels for sm_103a behind the
C ABI in ``include/attn_gqa.h``); this package is its Python binding, with the
same entry-point names, plus a few allocating helpers.  PyTorch supplies
device memory and streams only.
"""
from ._binding import (ATTN_BF16, ATTN_CAUSAL, ATTN_CROSS, ATTN_ERR_CUDA, ATTN_ERR_INVALID_ARG,  # noqa: F401
                       ATTN_ERR_TIMEOUT, ATTN_ERR_UNSUPPORTED, ATTN_FP32, ATTN_FULL, ATTN_OK, ATTN_TF32,
                       LIB_PATH, AttnError, attn_backward, attn_backward_rope, attn_decode_append, attn_decode_cached, attn_decode_cached_noalloc,
                       attn_decode_cached_window, attn_decode_paged, attn_decode_workspace_bytes, attn_forward, attn_forward_rope, attn_forward_window,
                       attn_get_status, attn_prefill, attn_prefill_paged, attn_prefill_window, attn_rope_table, attn_selftest_wait_timeout,
                       attn_status_string, load_library, attn_set_workspace, attn_forward_workspace_bytes,
                       attn_prefill_workspace_bytes, attn_backward_workspace_bytes, attn_scratch_reserved_bytes,
                       attn_scratch_peak_bytes, attn_release_scratch)
from .api import backward, decode, forward, prefill, rope_table, DecodeState  # noqa: F401
