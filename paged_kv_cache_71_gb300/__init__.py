"""Paged KV-cache decode for GB300 (sm_103a): a C-ABI CUDA library plus a thin binding.

The library (libpkv.so, built from csrc/) has the kernels; this package only
marshals arguments to it (``_binding``), builds seeded synthetic workloads
with a host block allocator (``workload``) and stages a workload on the
device to run one decode step (``runner``).
"""
from ._binding import (CacheDesc, PkvError, PKV_BF16, PKV_F32, PKV_FP8_E4M3, declared_entry_points, lib,
                       pkv_abi_version, pkv_block_hashes, pkv_copy_blocks, pkv_last_error, pkv_paged_attention_decode,
                       pkv_paged_attention_decode_shared, pkv_paged_attention_mixed,
                       pkv_paged_attention_mixed_workspace_size, pkv_paged_attention_decode_static_scratch,
                       pkv_paged_attention_workspace_size, pkv_paged_prefill_chunk, pkv_paged_prefill_varlen, pkv_reshape_and_cache,
                       pkv_status_string, pkv_swap_blocks)

__all__ = ["CacheDesc", "PkvError", "PKV_BF16", "PKV_F32", "PKV_FP8_E4M3", "declared_entry_points", "lib",
           "pkv_abi_version", "pkv_block_hashes", "pkv_copy_blocks", "pkv_last_error", "pkv_paged_attention_decode", "pkv_paged_attention_decode_shared",
           "pkv_paged_attention_mixed", "pkv_paged_attention_mixed_workspace_size", "pkv_paged_attention_decode_static_scratch",
           "pkv_paged_attention_workspace_size", "pkv_paged_prefill_chunk", "pkv_paged_prefill_varlen", "pkv_reshape_and_cache",
           "pkv_status_string", "pkv_swap_blocks"]
