"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every function here forwards to the C ABI with the same name (minus the
``pkv_`` prefix); all work happens in the library's CUDA kernels or its host
allocator. Tensors are passed as raw pointers (``tensor.data_ptr()``), the
stream as ``torch.cuda.current_stream().cuda_stream`` unless one is given.
If ``libpkv.so`` is missing the import fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "OUT_OF_BLOCKS", 3: "BAD_BLOCK", 4: "REFCOUNT", 5: "CUDA",
                6: "UNSUPPORTED"}
LAYOUTS = {"NHD": 0, "HND": 1}
KV_DTYPES = {"f16": 0, "e4m3": 1}
DEV_BAD_BLOCK, DEV_BAD_LENGTH, DEV_TIMEOUT, DEV_BAD_SLOT, DEV_BAD_PAIR = 0x1, 0x2, 0x4, 0x8, 0x10

EXPORTED = [
    "pkv_last_error", "pkv_version", "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_info", "pkv_alloc",
    "pkv_incref", "pkv_free", "pkv_refcount", "pkv_get_stats", "pkv_free_queue", "pkv_validate",
    "pkv_prepare_append", "pkv_append", "pkv_copy_blocks", "pkv_decode_attention", "pkv_decode_workspace_bytes",
    "pkv_pool_decode_attention", "pkv_decode_launch_info", "pkv_decode_append_attention",
    "pkv_decode_attention_static", "pkv_block_hash", "pkv_prompt_block_hashes", "pkv_prefix_lookup", "pkv_prefix_register",
    "pkv_pool_set_scales", "pkv_swap_bytes_per_block", "pkv_gather_blocks", "pkv_scatter_blocks",
    "pkv_prefill_attention", "pkv_cascade_plan", "pkv_prefix_pieces_bytes", "pkv_prefix_splits",
    "pkv_prefix_attention", "pkv_decode_attention_ex", "pkv_check_wait_limit",
]

MAX_GROUP_SEQS = 128
ATTN_INPUTS_EARLY = 0x1
ATTN_LAST_ROW_PENDING = 0x2
MAX_PREFIX_SPLITS = 8


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.code = STATUS_NAMES.get(status, str(status))


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("layout", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32)]


class PrefixGroup(ctypes.Structure):
    _fields_ = [("first_seq", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("prefix_tokens", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class Stats(ctypes.Structure):
    _fields_ = [("free_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32), ("shared_blocks", ctypes.c_int32),
                ("max_refcount", ctypes.c_int32), ("cow_copies", ctypes.c_int64), ("cached_blocks", ctypes.c_int32),
                ("cached_free_blocks", ctypes.c_int32), ("prefix_hits", ctypes.c_int64),
                ("prefix_misses", ctypes.c_int64), ("evictions", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_lib = None
vp, i32, i64, u64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run paged_kv_cache_88_gb300.build.build() "
                              "(the CUDA library is required, there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "pkv_last_error": (ctypes.c_char_p, []),
            "pkv_version": (i32, []),
            "pkv_pool_create": (i32, [ctypes.POINTER(PoolDesc), vp, vp, vp, ctypes.POINTER(vp)]),
            "pkv_pool_destroy": (i32, [vp]),
            "pkv_pool_info": (i32, [vp, ctypes.POINTER(PoolDesc), ctypes.POINTER(vp), ctypes.POINTER(vp)]),
            "pkv_alloc": (i32, [vp, i32, vp]),
            "pkv_incref": (i32, [vp, vp, i32]),
            "pkv_free": (i32, [vp, vp, i32]),
            "pkv_refcount": (i32, [vp, i32, ctypes.POINTER(i32)]),
            "pkv_get_stats": (i32, [vp, ctypes.POINTER(Stats)]),
            "pkv_free_queue": (i32, [vp, vp, i32, ctypes.POINTER(i32)]),
            "pkv_validate": (i32, [vp]),
            "pkv_prepare_append": (i32, [vp, i32, vp, i32, vp, vp, vp, i32, ctypes.POINTER(i32), vp, i32,
                                         ctypes.POINTER(i32)]),
            "pkv_append": (i32, [vp, i32, vp, vp, vp, i32, vp, vp]),
            "pkv_copy_blocks": (i32, [vp, vp, i32, vp, vp]),
            "pkv_decode_attention": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, i32, f32, vp, vp, sz,
                                           vp]),
            "pkv_decode_workspace_bytes": (sz, [i32, i32, i32]),
            "pkv_check_wait_limit": (i32, [vp, vp]),
            "pkv_pool_decode_attention": (i32, [vp, i32, vp, vp, i32, vp, i32, f32, vp, vp, sz, vp]),
            "pkv_decode_launch_info": (i32, [i32, i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                             ctypes.POINTER(i32)]),
            "pkv_decode_append_attention": (i32, [vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, f32, vp, vp, sz, vp]),
            "pkv_decode_attention_static": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, i32, vp, i32, f32, vp,
                                                  vp, vp]),
            "pkv_block_hash": (u64, [u64, vp, i32]),
            "pkv_prompt_block_hashes": (i32, [vp, i32, i32, vp, i32, ctypes.POINTER(i32)]),
            "pkv_prefix_lookup": (i32, [vp, vp, i32, vp, ctypes.POINTER(i32)]),
            "pkv_prefix_register": (i32, [vp, vp, vp, i32]),
            "pkv_pool_set_scales": (i32, [vp, vp, vp]),
            "pkv_swap_bytes_per_block": (sz, [vp]),
            "pkv_gather_blocks": (i32, [vp, vp, i32, vp, vp, vp]),
            "pkv_scatter_blocks": (i32, [vp, vp, i32, vp, vp, vp]),
            "pkv_prefill_attention": (i32, [vp, i32, vp, vp, i32, i32, i32, vp, i32, vp, f32, vp, vp, vp]),
            "pkv_cascade_plan": (i32, [vp, i32, vp, i32, i32, i32, i32, vp, i32, ctypes.POINTER(i32), vp]),
            "pkv_prefix_pieces_bytes": (sz, [i32, i32, i32]),
            "pkv_prefix_splits": (i32, [i32, i32, i32]),
            "pkv_prefix_attention": (i32, [vp, i32, vp, vp, i32, i32, vp, i32, i32, f32, vp, sz, vp,
                                           ctypes.c_uint32, vp]),
            "pkv_decode_attention_ex": (i32, [vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, vp, vp, i32, f32, vp, vp,
                                              sz, ctypes.c_uint32, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().pkv_last_error().decode()


def check(status: int) -> None:
    if status != OK:
        raise PkvError(status, last_error())


def _ptr(a) -> Optional[int]:
    """Address of a numpy array or torch tensor (None stays None)."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return a.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _require(t, dtype_name: str, what: str):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{what} must be a contiguous CUDA tensor")
    if str(t.dtype) != f"torch.{dtype_name}":
        raise ValueError(f"{what} must be {dtype_name}, got {t.dtype}")


class Pool:
    """A block pool (host metadata in libpkv) over caller-owned K/V pool tensors.

    ``k_pool``/``v_pool``: CUDA tensors of L*N*B*H*D elements (fp16, or uint8 E4M3
    codes for ``kv_dtype="e4m3"``) laid out as [L, N, H, B, D] (HND, the default) or
    [L, N, B, H, D] (NHD), or None for a host-only pool. ``k_scale``/``v_scale``
    (E4M3): fp32 tensors of L*N*H*B row scales, [L, N, H, B] in either layout.
    """

    def __init__(self, num_layers: int, num_blocks: int, block_size: int, num_heads: int, head_dim: int,
                 layout: str = "HND", k_pool=None, v_pool=None, initial_free_order: Optional[Sequence[int]] = None,
                 kv_dtype: str = "f16", k_scale=None, v_scale=None):
        self.desc = PoolDesc(num_layers, num_blocks, block_size, num_heads, head_dim, LAYOUTS[layout],
                             KV_DTYPES[kv_dtype])
        self.layout = layout
        self.kv_dtype = kv_dtype
        self.k_pool, self.v_pool = k_pool, v_pool
        self.k_scale, self.v_scale = k_scale, v_scale
        if k_pool is not None:
            el = "float16" if kv_dtype == "f16" else "uint8"
            _require(k_pool, el, "k_pool")
            _require(v_pool, el, "v_pool")
            want = num_layers * num_blocks * block_size * num_heads * head_dim
            if k_pool.numel() != want or v_pool.numel() != want:
                raise ValueError(f"pool tensors must hold {want} elements")
        order = None
        if initial_free_order is not None:
            order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
            if order.shape != (num_blocks,):
                raise ValueError("initial_free_order must have num_blocks entries")
        h = vp()
        check(lib().pkv_pool_create(ctypes.byref(self.desc), _ptr(k_pool), _ptr(v_pool), _ptr(order),
                                    ctypes.byref(h)))
        self._h = h
        if k_scale is not None:
            _require(k_scale, "float32", "k_scale")
            _require(v_scale, "float32", "v_scale")
            want = num_layers * num_blocks * num_heads * block_size
            if k_scale.numel() != want or v_scale.numel() != want:
                raise ValueError(f"scale pools must hold {want} elements")
            check(lib().pkv_pool_set_scales(self._h, _ptr(k_scale), _ptr(v_scale)))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().pkv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # -- host allocator ---------------------------------------------------------------
    def alloc(self, n: int) -> list:
        out = np.zeros(max(n, 1), dtype=np.int32)
        check(lib().pkv_alloc(self._h, n, _ptr(out)))
        return out[:n].tolist()

    def incref(self, ids: Sequence[int]) -> None:
        a = np.ascontiguousarray(ids, dtype=np.int32)
        check(lib().pkv_incref(self._h, _ptr(a), a.size))

    def free(self, ids: Sequence[int]) -> None:
        a = np.ascontiguousarray(ids, dtype=np.int32)
        check(lib().pkv_free(self._h, _ptr(a), a.size))

    def prefix_lookup(self, hashes: Sequence[int]) -> list:
        """Blocks of the longest cached run of ``hashes`` (each gets one more reference)."""
        h = np.ascontiguousarray(hashes, dtype=np.uint64)
        out = np.zeros(max(h.size, 1), dtype=np.int32)
        nh = i32()
        check(lib().pkv_prefix_lookup(self._h, _ptr(h), h.size, _ptr(out), ctypes.byref(nh)))
        return out[: nh.value].tolist()

    def prefix_register(self, hashes: Sequence[int], ids: Sequence[int]) -> None:
        h = np.ascontiguousarray(hashes, dtype=np.uint64)
        b = np.ascontiguousarray(ids, dtype=np.int32)
        if h.size != b.size:
            raise ValueError("one id per hash")
        check(lib().pkv_prefix_register(self._h, _ptr(h), _ptr(b), h.size))

    def refcount(self, block: int) -> int:
        r = i32()
        check(lib().pkv_refcount(self._h, block, ctypes.byref(r)))
        return r.value

    def stats(self) -> dict:
        s = Stats()
        check(lib().pkv_get_stats(self._h, ctypes.byref(s)))
        return s.as_dict()

    def free_queue(self) -> list:
        n = i32()
        out = np.zeros(self.desc.num_blocks, dtype=np.int32)
        check(lib().pkv_free_queue(self._h, _ptr(out), out.size, ctypes.byref(n)))
        return out[: n.value].tolist()

    def validate(self) -> None:
        check(lib().pkv_validate(self._h))

    def prepare_append(self, block_tables: np.ndarray, context_lens: np.ndarray,
                       num_new: Optional[Sequence[int]] = None,
                       slot_out: Optional[np.ndarray] = None, pair_out: Optional[np.ndarray] = None
                       ) -> Tuple[np.ndarray, np.ndarray]:
        """Host step a3; ``block_tables`` (int32 [S, maxb]) and ``context_lens`` (int32 [S]) change in place.

        Returns (slot_mapping int64 [n_tokens], copy_pairs int32 [n_pairs, 2]); with
        ``slot_out``/``pair_out`` given (e.g. pinned buffers) they are filled and views returned.
        """
        assert block_tables.dtype == np.int32 and block_tables.flags.c_contiguous
        assert context_lens.dtype == np.int32 and context_lens.flags.c_contiguous
        S, maxb = block_tables.shape
        nn = None if num_new is None else np.ascontiguousarray(num_new, dtype=np.int32)
        total = S if nn is None else int(nn.sum())
        slots = slot_out if slot_out is not None else np.zeros(max(total, 1), dtype=np.int64)
        pairs = pair_out if pair_out is not None else np.zeros((max(total, 1), 2), dtype=np.int32)
        ns, npair = i32(), i32()
        check(lib().pkv_prepare_append(self._h, S, _ptr(block_tables), maxb, _ptr(context_lens), _ptr(nn),
                                       _ptr(slots), slots.shape[0], ctypes.byref(ns), _ptr(pairs), pairs.shape[0],
                                       ctypes.byref(npair)))
        return slots[: ns.value], pairs[: npair.value]

    # -- device ops ---------------------------------------------------------------------
    def append(self, layer: int, k_new, v_new, slot_mapping, num_tokens: Optional[int] = None, status=None,
               stream=None) -> None:
        _require(k_new, "float16", "k_new")
        _require(v_new, "float16", "v_new")
        _require(slot_mapping, "int64", "slot_mapping")
        n = slot_mapping.numel() if num_tokens is None else num_tokens
        check(lib().pkv_append(self._h, layer, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n, _ptr(status),
                               _stream(stream)))

    def copy_blocks(self, pairs, num_pairs: Optional[int] = None, status=None, stream=None) -> None:
        _require(pairs, "int32", "pairs")
        n = pairs.numel() // 2 if num_pairs is None else num_pairs
        check(lib().pkv_copy_blocks(self._h, _ptr(pairs), n, _ptr(status), _stream(stream)))

    def decode_attention(self, layer: int, q, block_tables, context_lens, out, workspace, scale: float = 0.0,
                         stream=None) -> None:
        _require(q, "float16", "q")
        _require(out, "float16", "out")
        _require(block_tables, "int32", "block_tables")
        _require(context_lens, "int32", "context_lens")
        S = q.shape[0]
        check(lib().pkv_pool_decode_attention(self._h, layer, _ptr(q), _ptr(block_tables), block_tables.shape[1],
                                              _ptr(context_lens), S, float(scale), _ptr(out), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _stream(stream)))

    def decode_append_attention(self, layer: int, q, k_new, v_new, slot_mapping, block_tables, context_lens, out,
                                workspace, scale: float = 0.0, stream=None) -> None:
        """Append one token per sequence and attend, in one launch (pkv_decode_append_attention)."""
        for t, dt, name in ((q, "float16", "q"), (k_new, "float16", "k_new"), (v_new, "float16", "v_new"),
                            (out, "float16", "out"), (slot_mapping, "int64", "slot_mapping"),
                            (block_tables, "int32", "block_tables"), (context_lens, "int32", "context_lens")):
            _require(t, dt, name)
        check(lib().pkv_decode_append_attention(
            self._h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), q.shape[0], float(scale), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream)))

    def swap_bytes_per_block(self) -> int:
        return int(lib().pkv_swap_bytes_per_block(self._h))

    def gather_blocks(self, blocks_dev, dst, status=None, stream=None) -> None:
        """Copy the listed blocks (device int32) of every layer into ``dst`` (device bytes, or
        pinned host bytes mapped into the device's address space)."""
        _require(blocks_dev, "int32", "blocks")
        check(lib().pkv_gather_blocks(self._h, _ptr(blocks_dev), blocks_dev.numel(), _ptr(dst), _ptr(status),
                                      _stream(stream)))

    def scatter_blocks(self, blocks_dev, src, status=None, stream=None) -> None:
        """Copy ``src`` (laid out as gather_blocks writes it) into the listed blocks."""
        _require(blocks_dev, "int32", "blocks")
        check(lib().pkv_scatter_blocks(self._h, _ptr(blocks_dev), blocks_dev.numel(), _ptr(src), _ptr(status),
                                       _stream(stream)))

    def prefill_attention(self, layer: int, q, q_start, max_chunk: int, block_tables, context_lens, out, status,
                          scale: float = 0.0, stream=None) -> None:
        """Causal attention of each sequence's newest chunk over its cache (pkv_prefill_attention)."""
        for t, dt, name in ((q, "float16", "q"), (out, "float16", "out"), (q_start, "int32", "q_start"),
                            (block_tables, "int32", "block_tables"), (context_lens, "int32", "context_lens"),
                            (status, "int32", "status")):
            _require(t, dt, name)
        check(lib().pkv_prefill_attention(self._h, layer, _ptr(q), _ptr(q_start), q.shape[0], q_start.numel() - 1,
                                          max_chunk, _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                          float(scale), _ptr(out), _ptr(status), _stream(stream)))

    def prefix_attention(self, layer: int, q, groups_dev, num_groups: int, splits: int, block_tables, pieces,
                         status, scale: float = 0.0, flags: int = 0, stream=None) -> None:
        """The cascade's prefix pass (pkv_prefix_attention); ``groups_dev``: device int32 [G, 4];
        ``flags`` = ATTN_INPUTS_EARLY lets the launch start reading before its predecessor ends."""
        for t, dt, name in ((q, "float16", "q"), (groups_dev, "int32", "groups"),
                            (block_tables, "int32", "block_tables"), (status, "int32", "status")):
            _require(t, dt, name)
        check(lib().pkv_prefix_attention(self._h, layer, _ptr(q), _ptr(groups_dev), num_groups, splits,
                                         _ptr(block_tables), block_tables.shape[1], q.shape[0], float(scale),
                                         _ptr(pieces), pieces.numel() * pieces.element_size(), _ptr(status),
                                         flags, _stream(stream)))

    def decode_attention_ex(self, layer: int, q, block_tables, context_lens, out, workspace, k_new=None, v_new=None,
                            slot_mapping=None, seq_begin=None, pieces=None, splits: int = 0, scale: float = 0.0,
                            flags: int = 0, stream=None) -> None:
        """pkv_decode_attention_ex: optional fused append, optional cascade (private half + merge);
        ``flags`` = ATTN_INPUTS_EARLY lets the launch start reading before its predecessor ends
        (| ATTN_LAST_ROW_PENDING when that predecessor is the layer's append)."""
        for t, dt, name in ((q, "float16", "q"), (out, "float16", "out"), (block_tables, "int32", "block_tables"),
                            (context_lens, "int32", "context_lens")):
            _require(t, dt, name)
        check(lib().pkv_decode_attention_ex(
            self._h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(block_tables),
            block_tables.shape[1], _ptr(context_lens), q.shape[0], _ptr(seq_begin), _ptr(pieces), int(splits),
            float(scale), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), int(flags),
            _stream(stream)))

    def layer_view(self, which: str, layer: int):
        t = self.k_pool if which == "k" else self.v_pool
        d = self.desc
        return t.view(d.num_layers, -1)[layer]


def block_hash(parent: int, token_ids: Sequence[int]) -> int:
    """pkv_block_hash: chained hash of one block's token ids."""
    t = np.ascontiguousarray(token_ids, dtype=np.int32)
    return int(lib().pkv_block_hash(parent, _ptr(t), t.size))


def prompt_block_hashes(token_ids: Sequence[int], block_size: int) -> list:
    """pkv_prompt_block_hashes: chained hashes of the full blocks of a prompt."""
    t = np.ascontiguousarray(token_ids, dtype=np.int32)
    cap = t.size // block_size if block_size > 0 else 0
    out = np.zeros(max(cap, 1), dtype=np.uint64)
    n = ctypes.c_int32(0)
    check(lib().pkv_prompt_block_hashes(_ptr(t), t.size, block_size, _ptr(out), cap, ctypes.byref(n)))
    return [int(x) for x in out[:n.value]]


def cascade_plan(block_tables: np.ndarray, context_lens: np.ndarray, block_size: int, min_group: int = 2,
                 min_prefix_tokens: int = 0, max_groups: Optional[int] = None, groups_out: Optional[np.ndarray] = None,
                 begin_out: Optional[np.ndarray] = None):
    """pkv_cascade_plan on host arrays: (groups int32 [G, 4], seq_begin int32 [S]).

    ``groups_out`` / ``begin_out`` (optional, e.g. pinned staging) receive the
    plan in place; the returned arrays are views of them.
    """
    tab = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    S = tab.shape[0]
    cap = S if max_groups is None else max_groups
    groups = groups_out if groups_out is not None else np.zeros((max(cap, 1), 4), dtype=np.int32)
    begin = begin_out if begin_out is not None else np.zeros(S, dtype=np.int32)
    if groups.dtype != np.int32 or begin.dtype != np.int32 or groups.shape[0] < cap or begin.shape[0] < S:
        raise ValueError("plan buffers too small or not int32")
    n = i32()
    check(lib().pkv_cascade_plan(_ptr(tab), tab.shape[1], _ptr(lens), S, block_size, min_group, min_prefix_tokens,
                                 _ptr(groups), cap, ctypes.byref(n), _ptr(begin)))
    return groups[: n.value], begin[:S]


def check_wait_limit(status, stream=None) -> None:
    """pkv_check_wait_limit: a probe whose wait runs out; ``status``: device int32 [>= 1]."""
    _require(status, "int32", "status")
    check(lib().pkv_check_wait_limit(_ptr(status), _stream(stream)))


def prefix_pieces_bytes(num_seqs: int, num_heads: int, head_dim: int) -> int:
    n = lib().pkv_prefix_pieces_bytes(num_seqs, num_heads, head_dim)
    if n == 0 and num_seqs > 0:
        raise PkvError(1, last_error())
    return int(n)


def prefix_splits(num_groups: int, num_heads: int, max_prefix_tokens: int) -> int:
    return int(lib().pkv_prefix_splits(num_groups, num_heads, max_prefix_tokens))


def decode_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int) -> int:
    n = lib().pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim)
    if n == 0:
        raise PkvError(1, last_error())
    return int(n)


def new_workspace(num_seqs: int, num_heads: int, head_dim: int, device="cuda"):
    """A zero-filled workspace tensor (uint8) for :func:`decode_attention`; its first 4 bytes are the status word."""
    import torch
    return torch.zeros(decode_workspace_bytes(num_seqs, num_heads, head_dim), dtype=torch.uint8, device=device)


def workspace_status(workspace) -> int:
    """Read the device status word (first 4 bytes) of a workspace (synchronises)."""
    return int(workspace[:4].view(dtype=__import__("torch").int32).item()) & 0xFFFFFFFF


def decode_attention(q, k_cache, v_cache, block_tables, context_lens, *, num_blocks: int, block_size: int,
                     layout: str = "HND", scale: float = 0.0, out=None, workspace=None, stream=None):
    """Paged decode attention on one layer's caches (pkv_decode_attention); returns ``out``."""
    import torch
    _require(q, "float16", "q")
    _require(k_cache, "float16", "k_cache")
    _require(v_cache, "float16", "v_cache")
    _require(block_tables, "int32", "block_tables")
    _require(context_lens, "int32", "context_lens")
    S, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = new_workspace(S, H, D, q.device)
    check(lib().pkv_decode_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), num_blocks, block_size, H, D,
                                     LAYOUTS[layout], _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                     S, float(scale), _ptr(out), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def decode_launch_info(num_seqs: int, head_dim: int, kv_dtype: str = "f16") -> dict:
    """Grid of the decode attention kernel for a cache of kv_dtype ("f16" or "e4m3")."""
    g, per, sms = i32(), i32(), i32()
    check(lib().pkv_decode_launch_info(num_seqs, head_dim, KV_DTYPES[kv_dtype] if kv_dtype in KV_DTYPES else -1,
                                       ctypes.byref(g), ctypes.byref(per), ctypes.byref(sms)))
    return {"grid_ctas": g.value, "ctas_per_sm": per.value, "num_sms": sms.value}
