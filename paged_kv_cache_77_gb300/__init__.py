"""GB300-native paged KV cache: slot_mapping writes and paged attention on sm_103a.

The compute lives in libpaged_kv.so (C ABI, include/paged_kv.h); this package is
the build step and a thin ctypes binding over it.
"""
from . import api
from .api import (BlockPool, block_num_fixed, block_num_full_offline, block_num_full_online,
                  build_block_table_arange, build_slot_mapping, decode_workspace_size,
                  kv_cache_write, mla_paged_decode, num_skipped_tokens, paged_attention_decode,
                  paged_attention_decode_static, paged_attention_prefill)

__all__ = ["api", "BlockPool", "block_num_fixed", "block_num_full_offline",
           "block_num_full_online", "build_block_table_arange", "build_slot_mapping",
           "decode_workspace_size", "kv_cache_write", "mla_paged_decode", "num_skipped_tokens",
           "paged_attention_decode", "paged_attention_decode_static", "paged_attention_prefill"]
