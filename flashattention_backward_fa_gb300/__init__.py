"""GB300-native (sm_103a) FlashAttention forward and backward.

The computation lives in libfa.so, a C-ABI CUDA library (include/fa.h); this
package is its thin Python binding plus the seeded input generator used by the
tests and the bench. The library is loaded on first use and its absence is an
error: there is no CPU path.
"""
from .binding import (FA_BF16, FA_BWD_DKDV, FA_BWD_DQ, FA_BWD_PREPROCESS, FA_DQ_ATOMIC, FA_DQ_DETERMINISTIC,
                      FA_DQ_ORDERED, FA_DQ_RECOMPUTE, FA_F16, FA_F32, FaError, FaStrides,
                      alloc_workspace, attention_backward, attention_forward, default_scale, fa_bwd, fa_bwd_host,
                      fa_bwd_host_buffer_size,
                      fa_bwd_noalloc, fa_bwd_stage, fa_bwd_workspace_size, fa_fwd, fa_get_device_status, fa_selftest_timeout,
                      fa_strerror, fa_varlen_bwd, fa_varlen_bwd_workspace_size, fa_varlen_fwd, flash_attn_func,
                      flash_attn_varlen_func, header_functions,
                      load_library, varlen_attention_backward, varlen_attention_forward)

__all__ = ["FA_BF16", "FA_BWD_DKDV", "FA_BWD_DQ", "FA_BWD_PREPROCESS", "FA_DQ_ATOMIC", "FA_DQ_DETERMINISTIC",
           "FA_DQ_ORDERED", "FA_DQ_RECOMPUTE", "FA_F16", "FA_F32", "FaError", "FaStrides",
           "alloc_workspace", "attention_backward", "attention_forward", "default_scale", "fa_bwd", "fa_bwd_host",
           "fa_bwd_host_buffer_size", "fa_bwd_noalloc", "fa_bwd_stage",
           "fa_bwd_workspace_size", "fa_fwd", "fa_get_device_status", "fa_selftest_timeout", "fa_strerror",
           "fa_varlen_bwd",
           "fa_varlen_bwd_workspace_size", "fa_varlen_fwd", "flash_attn_func", "flash_attn_varlen_func", "header_functions", "load_library",
           "varlen_attention_backward", "varlen_attention_forward"]
