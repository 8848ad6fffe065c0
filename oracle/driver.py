"""Oracle replay of a workload: the allocator oracle plus float64 attention (test infrastructure only).

Mirrors a decode step of the product path with the oracle's own pieces:
``RefPool.prepare_append`` (slots, COW pairs), ``copy_blocks``, ``append_kv`` and
``decode_attention`` over NumPy pools. Shares nothing with the CUDA library; it
reads the same seeded inputs from ``workloads``.
"""
from __future__ import annotations

from typing import Callable, List, Optional

import numpy as np

import workloads as wl

from . import fp8
from . import ref_alloc as ra
from . import ref_attn as rf


class OracleEngine:
    def __init__(self, w: wl.Workload, k_pool: np.ndarray, v_pool: np.ndarray, k_scale=None, v_scale=None):
        """``k_pool``/``v_pool``: the initial pools, shape ``workloads.pool_shape(w)`` (copied); for an E4M3
        cache they are the codes and ``k_scale``/``v_scale`` the per-(token, head) scales."""
        self.w = w
        self.q8 = w.kv_dtype == "e4m3"
        dt = np.uint8 if self.q8 else np.float16
        self.k_pool = np.array(k_pool, dtype=dt, copy=True)
        self.v_pool = np.array(v_pool, dtype=dt, copy=True)
        self.k_scale = np.array(k_scale, dtype=np.float32, copy=True) if self.q8 else None
        self.v_scale = np.array(v_scale, dtype=np.float32, copy=True) if self.q8 else None
        self.pool = ra.RefPool(w.num_blocks, [int(x) for x in w.free_order])
        self.tables: List[List[int]] = [[-1] * w.max_blocks for _ in range(w.num_seqs)]
        self.lens: List[int] = [0] * w.num_seqs
        self.dummies = {}
        self.last_slots: list = []
        self.last_pairs: list = []

    def tables_array(self) -> np.ndarray:
        return np.asarray(self.tables, dtype=np.int32)

    def _copy(self, pairs):
        if self.q8:
            fp8.copy_blocks(self.k_pool, self.v_pool, self.k_scale, self.v_scale, pairs)
        else:
            rf.copy_blocks(self.k_pool, self.v_pool, pairs)

    def _append(self, layer, k_new, v_new, slots):
        if self.q8:
            fp8.append_kv(self.k_pool[layer], self.v_pool[layer], self.k_scale[layer], self.v_scale[layer], k_new,
                          v_new, slots, self.w.block_size, self.w.layout)
        else:
            rf.append_kv(self.k_pool[layer], self.v_pool[layer], k_new, v_new, slots, self.w.block_size,
                         self.w.layout)

    def run_script(self, values: Optional[Callable] = None):
        """Replay the set-up script. ``values(op_index, layer, which, n)`` gives written K/V (default: workloads)."""
        w, B = self.w, self.w.block_size
        values = values or (lambda oi, l, wh, n: wl.write_values(w, oi, l, wh, n))
        for op_index, op in enumerate(w.script):
            kind = op[0]
            if kind == "admit":
                _, s, T = op
                self.tables[s] = ra.admit(self.pool, T, B, w.max_blocks)
                self.lens[s] = T
            elif kind == "fork":
                _, src, dst = op
                self.tables[dst] = ra.fork(self.pool, self.tables[src], self.lens[src], B)
                self.lens[dst] = self.lens[src]
            elif kind == "dummy_alloc":
                _, d, n = op
                self.dummies[d] = self.pool.alloc(n)
            elif kind == "dummy_free":
                _, d = op
                self.pool.free(self.dummies.pop(d))
            elif kind == "write":
                counts = [int(x) for x in op[1]]
                total = sum(counts)
                slots, pairs = self.pool.prepare_append(self.tables, self.lens, counts, B, w.max_blocks)
                self._copy(pairs)
                for layer in range(w.num_layers):
                    self._append(layer, values(op_index, layer, 0, total), values(op_index, layer, 1, total), slots)
                self.last_slots, self.last_pairs = slots, pairs
            elif kind == "prompt":
                _, s, tokens = op
                hashes = ra.prompt_block_hashes(tokens, B)
                hit = self.pool.prefix_lookup(hashes)
                self.tables[s] = hit + [-1] * (w.max_blocks - len(hit))
                self.lens[s] = len(hit) * B
                counts = [0] * w.num_seqs
                counts[s] = len(tokens) - len(hit) * B
                total = counts[s]
                slots, pairs = self.pool.prepare_append(self.tables, self.lens, counts, B, w.max_blocks)
                self._copy(pairs)
                for layer in range(w.num_layers):
                    self._append(layer, values(op_index, layer, 0, total), values(op_index, layer, 1, total), slots)
                if len(hashes) > len(hit):
                    self.pool.prefix_register(hashes[len(hit):], self.tables[s][len(hit):len(hashes)])
                self.last_slots, self.last_pairs = slots, pairs
            else:
                raise ValueError(kind)

    def swap_out(self, s: int):
        """Copy sequence s's blocks (every layer) out and release them; returns the copies."""
        B = self.w.block_size
        n = -(-self.lens[s] // B)
        ids = self.tables[s][:n]
        saved = [a[:, ids].copy() for a in self._arrays()]
        self.pool.free(ids)
        self.tables[s] = [-1] * self.w.max_blocks
        return saved

    def swap_in(self, s: int, saved) -> None:
        """Allocate fresh blocks for sequence s and write the copies back into them."""
        n = saved[0].shape[1]
        ids = self.pool.alloc(n)
        self.tables[s] = ids + [-1] * (self.w.max_blocks - n)
        for a, v in zip(self._arrays(), saved):
            a[:, ids] = v

    def _arrays(self):
        return [self.k_pool, self.v_pool] + ([self.k_scale, self.v_scale] if self.q8 else [])

    def step(self, q: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, scale: Optional[float] = None,
             layers: Optional[list] = None, pairs_only: Optional[list] = None, impl: str = "numpy") -> np.ndarray:
        """One decode step: a3 (slots, COW), a4 copy, a5 append, a6/a7 attention. Returns float64 [L, S, H, D].

        ``impl="c"`` computes the attention with the C oracle (same definition,
        for full-size cases).
        """
        w = self.w
        slots, pairs = self.pool.prepare_append(self.tables, self.lens, [1] * w.num_seqs, w.block_size,
                                                w.max_blocks)
        self._copy(pairs)
        out = np.zeros((w.num_layers, w.num_seqs, w.num_heads, w.head_dim))
        tab = self.tables_array()
        for layer in range(w.num_layers):
            self._append(layer, k_new[layer], v_new[layer], slots)
            if layers is not None and layer not in layers:
                continue
            if self.q8:
                out[layer] = fp8.decode_attention(q[layer], self.k_pool[layer], self.v_pool[layer],
                                                  self.k_scale[layer], self.v_scale[layer], tab, self.lens,
                                                  w.block_size, scale, w.layout)
            elif impl == "c":
                from . import ref_attn_c as rc
                out[layer] = rc.decode_attention(q[layer], self.k_pool[layer], self.v_pool[layer], tab,
                                                 np.asarray(self.lens, dtype=np.int32), w.block_size, w.layout,
                                                 scale, pairs=pairs_only)
            else:
                out[layer] = rf.decode_attention(q[layer], self.k_pool[layer], self.v_pool[layer], tab, self.lens,
                                                 w.block_size, w.layout, scale, pairs=pairs_only)
        self.last_slots, self.last_pairs = slots, pairs
        return out

    def step_inputs(self, step: int):
        w = self.w
        q = np.stack([wl.query_values(w, step, l) for l in range(w.num_layers)])
        k = np.stack([wl.new_token_values(w, step, l, 0) for l in range(w.num_layers)])
        v = np.stack([wl.new_token_values(w, step, l, 1) for l in range(w.num_layers)])
        return q, k, v
