"""Paged KV-cache kernels for NVIDIA GB300 (sm_103a).

The compute lives in libpkv.so (CUDA kernels behind the C ABI of
include/pkv.h); ``pkv`` is its ctypes binding.  Build with
``paged_kv_cache_num_gb300.build.build()``.
"""
from .pkv import (KVCache, PkvError, copy_peak, decode_launches, decode_step, decode_workspace_bytes,
                  kv_append,
                  kv_append_scaled, lib, pack3, paged_decode, paged_decode_noalloc, slot_mapping,
                  unpack3, unpack3_words, version)

__all__ = ["KVCache", "PkvError", "copy_peak", "decode_launches", "decode_step", "decode_workspace_bytes",
           "kv_append", "kv_append_scaled", "lib", "pack3", "paged_decode", "paged_decode_noalloc", "slot_mapping",
           "unpack3", "unpack3_words", "version"]
