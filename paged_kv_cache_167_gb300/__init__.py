"""Paged KV-cache attention for one GB300 (sm_103a).

The product is the C-ABI library ``libpa.so`` (``include/pa.h``); this package
holds its CUDA sources (``csrc/``), the build script and a thin ctypes
binding with the same names.
"""
from .binding import (PA_DECODE_EARLY_METADATA, PA_SWAP_IN, PA_SWAP_OUT, PagedAttentionError, block_layout,
                      capacity_estimate, cascade_plan, check_wait_timeout, copy_blocks, decode, decode_cascade,
                      decode_grouped, decode_host, decode_host_staging_size, decode_noalloc, decode_partition_tokens,
                      decode_workspace_size, get_device_error, lib, pool_desc, prefill_chunk, prefix_attention,
                      reshape_and_cache, set_prefill_ctas, set_stream_k_ctas, slot_mapping, swap_blocks)
from .block_manager import BlockManager

__all__ = ["PagedAttentionError", "BlockManager", "PA_DECODE_EARLY_METADATA", "PA_SWAP_IN", "PA_SWAP_OUT",
           "block_layout", "capacity_estimate", "cascade_plan", "check_wait_timeout", "copy_blocks", "decode",
           "decode_cascade", "decode_grouped", "decode_host", "decode_host_staging_size", "decode_noalloc", "decode_partition_tokens",
           "decode_workspace_size", "get_device_error", "lib", "pool_desc", "prefill_chunk", "prefix_attention",
           "reshape_and_cache", "set_prefill_ctas", "set_stream_k_ctas", "slot_mapping", "swap_blocks"]
