"""GB300 (sm_103a) MLA decode over a paged latent KV cache.

Three CUDA kernels behind a C ABI (``include/mla_decode.h``): a tile scheduler
that partitions variable-length sequences into split-KV parts, the split-KV
attention kernel (bf16 cache, or packed e4m3 pages with per-token scales), and
an LSE-weighted combine.  This package is the thin
Python binding (``api``), the in-tree build (``build``) and the seeded
workload generator (``workloads``).
"""
from .api import (flash_mla_with_kvcache, get_mla_metadata, mla_decode_kvcache, mla_decode_kvcache_fp8,
                  mla_decode_kvcache_noalloc, mla_decode_kvcache_sparse, mla_device_status, mla_get_metadata,
                  mla_get_metadata_sparse, mla_num_sm_parts,
                  mla_set_cluster_multicast, mla_set_timing_events, mla_workspace_bytes)

__all__ = ["mla_get_metadata", "mla_get_metadata_sparse", "mla_decode_kvcache", "mla_decode_kvcache_fp8",
           "mla_decode_kvcache_sparse", "mla_decode_kvcache_noalloc",
           "mla_num_sm_parts", "mla_workspace_bytes", "mla_device_status", "mla_set_timing_events",
           "mla_set_cluster_multicast",
           "get_mla_metadata", "flash_mla_with_kvcache"]
