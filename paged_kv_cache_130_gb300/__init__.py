"""Paged KV-cache decode path for GB300 (sm_103a).

The compute runs in the CUDA library ``libpkv.so`` built from ``csrc/`` (see
``build.py``); ``binding`` is its thin ctypes front with the C entry-point
names, ``block_manager`` the host block allocator and ``workloads`` the seeded
workload generator.
"""
from .binding import (  # noqa: F401
    CacheDesc, PkvError, cache_desc, pkv_block_hashes, pkv_copy_blocks,
    pkv_decode_partition_size, pkv_decode_workspace_bytes, pkv_kv_append, pkv_lse_reduce,
    pkv_paged_attention_decode, pkv_paged_attention_decode_shared_prefix,
    pkv_paged_attention_decode_static_ws, pkv_paged_attention_partitions,
    pkv_paged_attention_prefill, pkv_shared_prefix_workspace_bytes, pkv_status_string,
    pkv_swap_blocks,
)
