"""ctypes front of the C attention oracle (test infrastructure only)."""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import numpy as np

from . import cbuild

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(cbuild.build())
        _lib.oracle_decode_attention.restype = ctypes.c_int
        _lib.oracle_decode_attention.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
        ]
        _lib.oracle_half_to_double.restype = ctypes.c_double
        _lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        _lib.oracle_max_threads.restype = ctypes.c_int
    return _lib


def max_threads() -> int:
    return lib().oracle_max_threads()


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(bits)


def decode_attention(q: np.ndarray, k_pool_layer: np.ndarray, v_pool_layer: np.ndarray,
                     block_tables: np.ndarray, context_lens: np.ndarray, block_size: int,
                     layout: str = "NHD", scale: Optional[float] = None,
                     pairs: Optional[Sequence[tuple]] = None, num_threads: int = 0) -> np.ndarray:
    """Same contract as ``ref_attn.decode_attention``; computed by the C loops."""
    S, H, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    q16 = np.ascontiguousarray(q, dtype=np.float16)
    k16 = np.ascontiguousarray(k_pool_layer, dtype=np.float16)
    v16 = np.ascontiguousarray(v_pool_layer, dtype=np.float16)
    N = k16.shape[0]
    B = block_size
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((S, H, D), dtype=np.float64)
    if pairs is not None:
        parr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        pptr, npairs = parr.ctypes.data, parr.shape[0]
    else:
        parr, pptr, npairs = None, None, 0
    rc = lib().oracle_decode_attention(
        q16.ctypes.data, k16.ctypes.data, v16.ctypes.data, 0 if layout == "NHD" else 1, N, B, H, D,
        tables.ctypes.data, tables.shape[1], lens.ctypes.data, S, float(scale), out.ctypes.data,
        pptr, npairs, num_threads)
    if rc == -2:
        raise MemoryError("C oracle ran out of scratch memory")
    if rc != 0:
        raise ValueError("C oracle rejected its arguments (block id or length out of range)")
    return out
