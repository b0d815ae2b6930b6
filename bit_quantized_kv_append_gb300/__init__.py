"""GB300-native low-bit KV-cache quantization for LLM decode.

The work runs in ``libkvq.so`` (hand-written sm_103a CUDA kernels behind the C
ABI of ``include/kvq.h``); this package only builds and binds it.
"""
from .kvq import (BUFFERS, EXPORTS, CacheRef, Config, KvqError, Layout, PagedCacheRef, PagedKVCache,
                  QuantizedKVCache, append, append_levels, append_window, decode_attn, decode_attn_diag,
                  decode_attn_levels, decode_attn_noalloc, decode_step, decode_step_levels, fit_levels, layout, lib,
                  make_config,
                  paged_append, paged_decode_attn, paged_layout, rope_init)

__all__ = ["BUFFERS", "EXPORTS", "CacheRef", "Config", "KvqError", "Layout", "PagedCacheRef", "PagedKVCache",
           "QuantizedKVCache", "append", "append_levels", "append_window", "decode_attn", "decode_attn_levels",
           "decode_attn_noalloc", "decode_attn_diag", "decode_step", "decode_step_levels", "fit_levels", "layout", "lib",
           "make_config", "paged_append", "paged_decode_attn", "paged_layout", "rope_init"]
