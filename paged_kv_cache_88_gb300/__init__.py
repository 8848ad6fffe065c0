"""paged_kv_cache_88_gb300 -- a paged KV cache and paged decode attention for GB300 (sm_103a).

The work is done by ``libpkv.so`` (C ABI in ``include/pkv.h``): a host block
allocator (FIFO free queue, refcounts, copy-on-write) and hand-written CUDA
kernels for the append scatter, the block copy and split-KV decode attention.
This package is the thin ctypes binding plus the decode-step driver used by the
tests and the benchmark. Importing it without the built library raises.
"""
from .binding import (DEV_BAD_BLOCK, DEV_BAD_LENGTH, DEV_BAD_PAIR, DEV_BAD_SLOT, DEV_TIMEOUT, EXPORTED, LAYOUTS,
                      PkvError, Pool, decode_attention, decode_launch_info, decode_workspace_bytes, last_error, lib,
                      new_workspace, workspace_status)

lib()  # fail loudly at import if the CUDA library is missing

__all__ = [
    "Pool", "PkvError", "decode_attention", "decode_workspace_bytes", "new_workspace", "workspace_status",
    "decode_launch_info", "last_error", "lib", "LAYOUTS", "EXPORTED", "DEV_BAD_BLOCK", "DEV_BAD_LENGTH",
    "DEV_TIMEOUT", "DEV_BAD_SLOT", "DEV_BAD_PAIR",
]
