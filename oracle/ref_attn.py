"""Decode-attention, append and block-copy oracle in float64 (NumPy).

Test infrastructure only (see ``oracle/__init__``).

The result is the plain definition, not the split-KV algorithm that reaches it:
for each sequence s and head h, gather the sequence's keys and values token by
token through its block table and compute ``softmax(scale * K q) V`` with the
maximum subtracted, all in float64. The pages fix this meaning:

* decode attends the current query over the whole cached history
  (icman.com.cn/news/78786 §1.1);
* the paged kernel walks the block table and loads each block's K/V
  (icman.com.cn/news/78786 §2.4);
* logical position p lives in physical page ``table[p // page_size]`` at slot
  ``p % page_size`` (m.lqnn.cn/news/240480 §3.3).

Pool layout (a reading; the pages print ``[page, slot, head, dim]`` in
m.lqnn.cn/news/240480 §3.3 but garble the offsets): each layer is an array of
``N`` blocks; a block holds ``B x H x D`` elements either as ``[B][H][D]``
("NHD", the page's order) or ``[H][B][D]`` ("HND"). Both lay out the same
block-sized bytes; :func:`kv_row` is the one place that maps (block, slot, head)
to a row of ``D`` contiguous elements, so every result here is layout-agnostic.

Other readings: scale defaults to ``1/sqrt(D)`` (the pages pass no scale);
an empty context (T = 0) gives a zero output; a slot < 0 is not written.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

LAYOUTS = ("NHD", "HND")


def kv_row(layout: str, block: int, slot: int, head: int, num_heads: int, block_size: int) -> int:
    """Row (of D elements) holding (block, slot, head) within one layer's pool."""
    if layout == "NHD":
        return (block * block_size + slot) * num_heads + head
    if layout == "HND":
        return (block * num_heads + head) * block_size + slot
    raise ValueError(f"unknown layout {layout!r}")


def layer_rows(pool_layer: np.ndarray, head_dim: int) -> np.ndarray:
    """View one layer's pool (any of the two block shapes) as rows of D elements."""
    return pool_layer.reshape(-1, head_dim)


def gather_sequence(pool_layer: np.ndarray, table_row: Sequence[int], num_tokens: int, head: int,
                    layout: str, num_heads: int, block_size: int, head_dim: int) -> np.ndarray:
    """K (or V) of one (sequence, head) as a contiguous float64 [T, D] array."""
    rows = layer_rows(pool_layer, head_dim)
    idx = [kv_row(layout, int(table_row[t // block_size]), t % block_size, head, num_heads, block_size)
           for t in range(num_tokens)]
    return rows[np.asarray(idx, dtype=np.int64)].astype(np.float64)


def softmax_weights(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """Attention weights of one query over T keys (float64, max-subtracted)."""
    x = scale * (k.astype(np.float64) @ q.astype(np.float64))
    x = x - x.max()
    w = np.exp(x)
    return w / w.sum()


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * k q) v for one query, contiguous k, v [T, D]; zeros if T = 0."""
    if k.shape[0] == 0:
        return np.zeros(v.shape[1], dtype=np.float64)
    return softmax_weights(q, k, scale) @ v.astype(np.float64)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def decode_attention(q: np.ndarray, k_pool_layer: np.ndarray, v_pool_layer: np.ndarray,
                     block_tables: np.ndarray, context_lens: Sequence[int], block_size: int,
                     layout: str = "NHD", scale: Optional[float] = None,
                     pairs: Optional[Sequence[tuple]] = None) -> np.ndarray:
    """Paged decode attention for one layer; returns float64 [S, H, D].

    ``q`` is [S, H, D]; the pools are one layer's blocks; ``block_tables`` is
    [S, max_blocks]. ``pairs`` restricts the work to the listed (s, h) pairs
    (other outputs stay zero) so that large cases can be sampled.
    """
    S, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    out = np.zeros((S, H, D), dtype=np.float64)
    todo = pairs if pairs is not None else [(s, h) for s in range(S) for h in range(H)]
    for s, h in todo:
        T = int(context_lens[s])
        k = gather_sequence(k_pool_layer, block_tables[s], T, h, layout, H, block_size, D)
        v = gather_sequence(v_pool_layer, block_tables[s], T, h, layout, H, block_size, D)
        out[s, h] = attend(q[s, h], k, v, scale)
    return out


def append_kv(k_pool_layer: np.ndarray, v_pool_layer: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
              slot_mapping: Sequence[int], block_size: int, layout: str = "NHD") -> None:
    """Write token i's K/V (all heads) to ``slot_mapping[i]`` in place; slot < 0 is skipped.

    m.lqnn.cn/news/240480 §3.2 step 3 gives the slot; the write is a bit copy.
    """
    n, H, D = k_new.shape
    k_rows = layer_rows(k_pool_layer, D)
    v_rows = layer_rows(v_pool_layer, D)
    for i in range(n):
        slot = int(slot_mapping[i])
        if slot < 0:
            continue
        block, offset = divmod(slot, block_size)
        for h in range(H):
            r = kv_row(layout, block, offset, h, H, block_size)
            k_rows[r] = k_new[i, h]
            v_rows[r] = v_new[i, h]


def copy_blocks(k_pool: np.ndarray, v_pool: np.ndarray, pairs: Sequence[tuple]) -> None:
    """Copy-on-write data move: block dst <- block src in every layer, K and V.

    ``k_pool``/``v_pool`` are [L, N, ...]; hnwysp.cn/news/103996 §3.3 copies the
    whole block before the new token is written into it.
    """
    for src, dst in pairs:
        k_pool[:, dst] = k_pool[:, src]
        v_pool[:, dst] = v_pool[:, src]


def prefill_attention(q: np.ndarray, k_pool_layer: np.ndarray, v_pool_layer: np.ndarray,
                      block_tables: np.ndarray, context_lens: Sequence[int], q_start: Sequence[int],
                      block_size: int, layout: str = "HND", scale: Optional[float] = None) -> np.ndarray:
    """Causal (prefill) attention of each sequence's newest chunk over its paged cache, float64.

    Sequence s's chunk is rows q_start[s] .. q_start[s+1]-1 of ``q`` ([rows, H, D]),
    its C_s tokens are the last C_s of its T_s = context_lens[s] cached tokens, and
    query i (position p = T_s - C_s + i) attends to cached tokens 0..p
    (m.lqnn.cn/news/240480 §3.3, §4.3). Returns [rows, H, D].
    """
    R, H, D = q.shape
    if scale is None:
        scale = default_scale(D)
    out = np.zeros((R, H, D), dtype=np.float64)
    for s in range(len(context_lens)):
        r0, r1 = int(q_start[s]), int(q_start[s + 1])
        C, T = r1 - r0, int(context_lens[s])
        if C == 0:
            continue
        pos = np.arange(T - C, T)
        for h in range(H):
            k = gather_sequence(k_pool_layer, block_tables[s], T, h, layout, H, block_size, D)
            v = gather_sequence(v_pool_layer, block_tables[s], T, h, layout, H, block_size, D)
            x = scale * (q[r0:r1, h].astype(np.float64) @ k.T)            # [C, T]
            x[np.arange(T)[None, :] > pos[:, None]] = -np.inf              # causal: keys after the query
            x = x - x.max(axis=1, keepdims=True)
            w = np.exp(x)
            w /= w.sum(axis=1, keepdims=True)
            out[r0:r1, h] = w @ v
    return out
