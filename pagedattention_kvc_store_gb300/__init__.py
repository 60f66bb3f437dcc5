"""Paged KV-cache store and paged attention for NVIDIA GB300 (sm_103a).

The product is the C-ABI library libkvc.so (include/kvc.h), built from ``csrc/`` by
``build.build()``; ``kvc`` is its thin Python binding (same entry-point names).
"""
from .kvc import (EXPORTS, KVC_BF16, KVC_F32, KVC_HND, KVC_NHD, NOALLOC_SCRATCH_BYTES, KvcError,
                  PoolDesc,
                  kvc_append, kvc_append_store, kvc_copy_pages, kvc_decode, kvc_decode_noalloc, kvc_decode_plan,
                  kvc_decode_store,
                  kvc_decode_shared_prefix, kvc_decode_shared_prefix_plan, kvc_shared_prefix_groups,
                  kvc_decode_int8, kvc_decode_int8_plan, kvc_decode_int8_store, kvc_append_int8,
                  kvc_device_errors, kvc_selftest_wait, kvc_set_error_word, kvc_merge,
                  kvc_slot_mapping, kvc_store, kvc_store_int8, int8_pool_desc,
                  kvc_validate, kvc_validate_workspace_size, lib, library_path, pool_desc)

__all__ = ["EXPORTS", "KVC_BF16", "KVC_F32", "KVC_HND", "KVC_NHD", "NOALLOC_SCRATCH_BYTES",
           "KvcError", "PoolDesc",
           "kvc_append", "kvc_append_store", "kvc_copy_pages", "kvc_decode", "kvc_decode_noalloc", "kvc_decode_plan",
           "kvc_decode_store",
           "kvc_decode_shared_prefix", "kvc_decode_shared_prefix_plan", "kvc_shared_prefix_groups",
           "kvc_decode_int8", "kvc_decode_int8_plan", "kvc_decode_int8_store", "kvc_append_int8",
           "kvc_device_errors", "kvc_selftest_wait", "kvc_set_error_word", "kvc_merge",
           "kvc_slot_mapping",
           "kvc_store", "kvc_store_int8", "int8_pool_desc",
           "kvc_validate", "kvc_validate_workspace_size", "lib", "library_path", "pool_desc"]
