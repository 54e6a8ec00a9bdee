"""paged_kv_cache_24_gb300 -- paged KV-cache decode attention for GB300 (sm_103a).

Public API (thin wrappers over the C ABI of ``libpkv.so``, see include/pkv.h):

* ``pkv_slot_mapping(block_tables, positions, block_size)`` -- slot of each
  sequence's new token;
* ``pkv_append(k, v, slot_mapping, k_cache, v_cache)`` -- write the new
  tokens' K/V into their slots;
* ``pkv_decode(q, k_cache, v_cache, block_tables, context_lens, window, scale,
  out)`` -- single-query attention over each sequence's paged context,
  optionally limited to a sliding window;
* ``pkv_append_decode(q, k_new, v_new, k_cache, v_cache, block_tables,
  context_lens, window, scale)`` -- both in one launch;
* ``pkv_append_fp8(k, v, slot_mapping, k_codes, v_codes, k_scale, v_scale)``
  and ``pkv_append_int8(...)`` -- quantising append into FP8 E4M3 (uint8) or
  INT8 (int8) pools, which ``pkv_decode`` reads when given the row scales;
* ``pkv_prefill(q, k, v, cu_q, k_cache, v_cache, block_tables, context_lens,
  window, scale, max_chunk, num_sinks=0)`` -- chunked prefill: append packed
  chunks and compute their causal (windowed, with sinks) attention over the
  paged cache;
* ``pkv_stage_copy(dst, src)`` -- a kernel copy between device memory and
  pinned host memory (DecodeStep's host transfers);
* ``pkv_device_address(t)`` -- the address the kernels use for a device or
  pinned host tensor (a decode may read q and the new K/V from, and write
  ``out`` to, pinned host memory);
* ``pkv_validate_indices(block_tables, context_lens, num_blocks, block_size,
  slot_mapping=None)`` -- debug check of the indices the kernels trust
  (waits for the stream).

``DecodeStep`` packages one serving step (slot mapping, append, decode) as a
CUDA graph fed from a pinned host staging buffer.

All tensors live on the GPU; PyTorch provides the memory and the stream.
``workloads`` builds the seeded synthetic inputs used by the tests and the
benchmark.
"""
from ._binding import (CacheLayout, DecodeOptions, PkvError, cache_layout, library_path, load_library,
                       pkv_append, pkv_append_decode, pkv_append_fp8, pkv_append_int8, pkv_decode, pkv_prefill, pkv_decode_plan, pkv_release_workspaces,
                       pkv_device_address, pkv_slot_mapping, pkv_stage_copy,
                       pkv_validate_indices, status_string,
                       PKV_ERR_RANGE, PKV_ERR_UNSUPPORTED)
from .step import DecodeStep

__all__ = [
    "DecodeStep", "DecodeOptions", "CacheLayout", "PkvError", "cache_layout", "library_path", "load_library", "pkv_append",
    "pkv_append_decode", "pkv_append_fp8", "pkv_append_int8", "pkv_prefill",
    "pkv_decode", "pkv_decode_plan", "pkv_release_workspaces", "pkv_slot_mapping", "pkv_stage_copy",
    "pkv_validate_indices", "pkv_device_address", "PKV_ERR_RANGE", "PKV_ERR_UNSUPPORTED",
    "status_string",
]
