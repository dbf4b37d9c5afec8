"""Paged-KV attention for GB300 (sm_103a): a thin Python face over the C ABI in include/pkv.h.

All work runs in the CUDA kernels of ``libpkv.so`` (built in-tree by
``paged_kv_cache_160_gb300/build.py``); this package only marshals torch tensors into
pointers.  Importing it without the built library raises ImportError.
"""
from ._binding import (  # noqa: F401
    BlockManager,
    CacheDesc,
    NoBlocksError,
    PkvError,
    DEVERR,
    cache_desc,
    lib,
    pkv_check_bounded_wait,
    pkv_copy_blocks,
    pkv_decode_workspace_bytes,
    pkv_get_device_error,
    pkv_kv_write,
    pkv_paged_decode,
    pkv_paged_decode_append,
    pkv_paged_decode_noalloc,
    pkv_noalloc_scratch_bytes,
    pkv_get_decode_sm_budget,
    pkv_set_decode_sm_budget,
    pkv_paged_prefill_chunk,
    pkv_stream_tiles,
    pkv_swap_blocks,
)
