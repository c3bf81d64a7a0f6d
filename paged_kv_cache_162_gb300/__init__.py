"""pagedkv: paged KV-cache decode attention for NVIDIA GB300 (sm_103a).

The library is libpagedkv.so (CUDA kernels + C ABI, include/pagedkv.h);
this package is its Python binding:
  _lib        ctypes binding, one function per C entry point, same names
  allocator   host block allocator (free list + per-block refcounts)
  engine      tensor-level calls and one decode step (DecodeStep)
"""
from ._lib import (PKV_BF16, PKV_F16, OutOfBlocks, PkvError, lib, pkv_compute_slot_mapping,
                   pkv_copy_blocks, pkv_decode_workspace_size, pkv_get_device_errors,
                   pkv_last_error_string, pkv_paged_attention_decode, pkv_reshape_and_cache,
                   pkv_sync_check, pkv_version)
from .allocator import BlockAllocator, plan_step

__all__ = [
    "PKV_BF16", "PKV_F16", "OutOfBlocks", "PkvError", "lib", "pkv_compute_slot_mapping",
    "pkv_copy_blocks", "pkv_decode_workspace_size", "pkv_get_device_errors",
    "pkv_last_error_string", "pkv_paged_attention_decode", "pkv_reshape_and_cache",
    "pkv_sync_check", "pkv_version", "BlockAllocator", "plan_step",
]
