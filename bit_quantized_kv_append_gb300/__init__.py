"""GB300-native low-bit KV-cache quantization for LLM decode.

The work runs in ``libkvq.so`` (hand-written sm_103a CUDA kernels behind the C
ABI of ``include/kvq.h``); this package only builds and binds it.
"""
from .kvq import (BUFFERS, EXPORTS, CacheRef, Config, KvqError, Layout, QuantizedKVCache, append,
                  decode_attn, decode_attn_noalloc, layout, lib, make_config, rope_init)

__all__ = ["BUFFERS", "EXPORTS", "CacheRef", "Config", "KvqError", "Layout", "QuantizedKVCache",
           "append", "decode_attn", "decode_attn_noalloc", "layout", "lib", "make_config", "rope_init"]
