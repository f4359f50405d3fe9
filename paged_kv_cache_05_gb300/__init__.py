"""GB300-native paged KV-cache decode path (PagedAttention) behind a C ABI.

The compute lives in libpagedkv.so (CUDA kernels for sm_103a plus the C++
block manager); ``pagedkv`` is its thin ctypes binding and ``workloads`` the
seeded synthetic inputs.  Build with ``python -m paged_kv_cache_05_gb300.build``.
"""
from .pagedkv import (BlockManager, OutOfBlocks, PagedKVError, alloc_workspace, copy_blocks,
                      contiguous_attention_decode, contiguous_workspace_size,
                      decode_shared_workspace_size, decode_workspace_size, get_device_error, lib, paged_attention_decode,
                      paged_attention_decode_append,
                      paged_attention_decode_noalloc, paged_attention_decode_shared,
                      paged_attention_prefill, paged_attention_prefill_write,
                      reshape_and_cache, set_decode_wait_limit, swap_blocks, version)

__all__ = ["BlockManager", "OutOfBlocks", "PagedKVError", "alloc_workspace", "copy_blocks",
           "contiguous_attention_decode", "contiguous_workspace_size",
           "decode_shared_workspace_size", "decode_workspace_size", "get_device_error", "lib", "paged_attention_decode",
           "paged_attention_decode_append",
           "paged_attention_decode_noalloc", "paged_attention_decode_shared",
           "paged_attention_prefill", "paged_attention_prefill_write",
           "reshape_and_cache", "set_decode_wait_limit", "swap_blocks", "version"]
