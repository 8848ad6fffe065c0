"""Closed-form sizes of a paged KV cache (oracle; test infrastructure only).

Each function restates a formula the pages print:

* bytes of K and V per token over all layers -- hnwysp.cn/news/103996 §1.2 and
  icman.com.cn/news/78786 §1.1: two matrices (K and V) x layers x hidden width
  (heads x head_dim) x bytes per element;
* bytes per token per layer and per page -- m.lqnn.cn/news/240480 §3.1;
* blocks in a pool and the concurrency it supports -- icman.com.cn/news/78786 §4.1:
  blocks = usable bytes / (block size x bytes per token);
* block-table entries -- icman.com.cn/news/78786 §2.2: one entry per started block;
* internal waste -- hnwysp.cn/news/103996 §3.1 and icman.com.cn/news/78786 §2.2:
  the unused tail of each sequence's last block, about half a block on average.
"""
from __future__ import annotations

from typing import Iterable


def kv_bytes_per_token(num_layers: int, hidden: int, dtype_bytes: int) -> int:
    """K and V bytes one token occupies across all layers (2 x L x hidden x bytes)."""
    return 2 * num_layers * hidden * dtype_bytes


def kv_bytes_per_token_layer(num_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """K and V bytes one token occupies in one layer (2 x heads x head_dim x bytes)."""
    return 2 * num_heads * head_dim * dtype_bytes


def block_bytes(block_tokens: int, bytes_per_token: int) -> int:
    """Bytes of one block (page) holding ``block_tokens`` tokens."""
    return block_tokens * bytes_per_token


def request_bytes(num_tokens: int, bytes_per_token: int) -> int:
    """KV bytes of one request of ``num_tokens`` tokens (no paging waste)."""
    return num_tokens * bytes_per_token


def pool_blocks(usable_bytes: int, block_tokens: int, bytes_per_token: int) -> int:
    """Whole blocks that fit in ``usable_bytes``."""
    return usable_bytes // block_bytes(block_tokens, bytes_per_token)


def pool_tokens(num_blocks: int, block_tokens: int) -> int:
    """Token capacity of a pool of ``num_blocks`` blocks."""
    return num_blocks * block_tokens


def max_concurrency(num_blocks: int, block_tokens: int, mean_tokens: int) -> int:
    """Requests of ``mean_tokens`` tokens that fit in the pool at once (floor)."""
    return pool_tokens(num_blocks, block_tokens) // mean_tokens


def table_entries(num_tokens: int, block_tokens: int) -> int:
    """Block-table entries a sequence of ``num_tokens`` tokens needs."""
    return -(-num_tokens // block_tokens)


def wasted_slots(num_tokens: int, block_tokens: int) -> int:
    """Unused token slots in the last block of one sequence."""
    return table_entries(num_tokens, block_tokens) * block_tokens - num_tokens


def internal_waste_fraction(lengths: Iterable[int], block_tokens: int) -> float:
    """Unused slots over used slots, summed over a set of sequences."""
    lengths = [int(t) for t in lengths]
    used = sum(lengths)
    if used == 0:
        return 0.0
    return sum(wasted_slots(t, block_tokens) for t in lengths) / used


def expected_waste_uniform_residue(block_tokens: int) -> float:
    """Mean unused slots when a length's residue mod B is uniform on 0..B-1.

    A residue r > 0 wastes B - r slots and r = 0 wastes none, so the mean is
    (B - 1) / 2: the "about half a block" of hnwysp.cn/news/103996 §3.1.
    """
    b = block_tokens
    return sum((b - r) % b for r in range(b)) / b


def gib(x: float) -> int:
    return int(round(x * (1 << 30)))


def mib(x: float) -> int:
    return int(round(x * (1 << 20)))


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)

