"""Block-pool oracle: FIFO free queue, refcounts, append-slot and copy-on-write.

Test infrastructure only (see ``oracle/__init__``). Pure Python, no arithmetic
shared with the product library.

What it follows:

* A pool is cut once into N fixed-size blocks and every block is threaded onto a
  free list (hnwysp.cn/news/103996 §3.2, §4.1; icman.com.cn/news/78786 §2.3).
* Blocks are taken from the head of the free queue and returned to its tail
  (hnwysp.cn/news/103996 §3.4). The initial order of the queue is an input (the
  pages start from ``arange``, m.lqnn.cn/news/240480 §4.2; the workloads pass a
  seeded permutation).
* Each block carries a refcount; a block shared by several sequences is returned
  to the free queue only when its count reaches zero (hnwysp.cn/news/103996 §3.3,
  §4.4; icman.com.cn/news/78786 §3.4, §6.3).
* A new token at position p of a sequence goes to logical block p // B, slot
  p % B; a fresh block is taken when the last one is full
  (m.lqnn.cn/news/240480 §3.2 step 3; icman.com.cn/news/78786 §2.3).
* Copy-on-write: writing into a block that other sequences still reference first
  takes a new block, copies the old block into it and writes there; only the
  block at the fork point is copied (hnwysp.cn/news/103996 §3.3;
  icman.com.cn/news/78786 §3.4).

* Prefix caching: each full block of a prompt is keyed by a hash of its tokens
  chained from the start of the sequence; a request whose leading blocks hash
  to cached blocks shares them (one more reference, no KV written); cached
  blocks with no reference stay evictable in LRU order and a later hit revives
  them (icman.com.cn/news/78786 §3.1-§3.4; hnwysp.cn/news/103996 §4.3).

Readings taken where the pages are silent:

* Allocation is all-or-nothing and a failed call changes nothing.
* COW fires iff the refcount of the block being written is > 1 at the moment of
  the write; sequences are processed in ascending index, tokens in order.
* A slot is ``physical_block * B + offset``; -1 in a table means "no block".
* The block hash is 64-bit FNV-1a (the pages name SHA256 or xxHash; any fixed
  hash serves) over the parent hash's 8 little-endian bytes and the block's
  token ids, 4 little-endian bytes each; the first block's parent is 0.
* The free queue is the LRU of cached blocks: a freed block keeps its hash at
  the tail; a hit takes it back out; reusing it from the head drops its hash.
  Lookup stops at the first miss (a chained hash past a miss cannot be used).
"""
from __future__ import annotations

import copy
from collections import deque
from dataclasses import dataclass
from typing import List, Optional, Sequence


class PoolError(Exception):
    """Raised by the oracle pool; ``code`` names the failure."""

    def __init__(self, code: str, msg: str = ""):
        super().__init__(f"{code}: {msg}")
        self.code = code


OUT_OF_BLOCKS = "out_of_blocks"
BAD_BLOCK = "bad_block"
REFCOUNT = "refcount"
INVALID_ARG = "invalid_arg"


FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """64-bit FNV-1a: xor each byte into the state, then multiply by the FNV prime."""
    h = FNV64_OFFSET
    for byte in data:
        h = ((h ^ byte) * FNV64_PRIME) & MASK64
    return h


def block_hash(parent: int, token_ids: Sequence[int]) -> int:
    """Hash of one block chained on its parent's hash (0 for the first block)."""
    data = int(parent).to_bytes(8, "little") + b"".join(int(t).to_bytes(4, "little", signed=True)
                                                       for t in token_ids)
    return fnv1a64(data)


def prompt_block_hashes(token_ids: Sequence[int], block_size: int) -> List[int]:
    """Chained hashes of the full blocks of a prompt."""
    out, parent = [], 0
    for i in range(len(token_ids) // block_size):
        parent = block_hash(parent, token_ids[i * block_size:(i + 1) * block_size])
        out.append(parent)
    return out


@dataclass
class PoolStats:
    free_blocks: int
    used_blocks: int
    shared_blocks: int
    max_refcount: int
    cow_copies: int
    cached_blocks: int = 0
    cached_free_blocks: int = 0
    prefix_hits: int = 0
    prefix_misses: int = 0
    evictions: int = 0


class RefPool:
    """N blocks, a FIFO free queue and a refcount per block."""

    def __init__(self, num_blocks: int, initial_free_order: Optional[Sequence[int]] = None):
        if num_blocks <= 0:
            raise PoolError(INVALID_ARG, "num_blocks must be positive")
        order = list(range(num_blocks)) if initial_free_order is None else [int(x) for x in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise PoolError(INVALID_ARG, "initial free order must be a permutation of 0..N-1")
        self.num_blocks = num_blocks
        self.free_queue: deque = deque(order)
        self.refcount: List[int] = [0] * num_blocks
        self.cow_copies = 0
        self.hash_of: dict = {}     # block -> registered hash
        self.by_hash: dict = {}     # hash -> block
        self.prefix_hits = 0
        self.prefix_misses = 0
        self.evictions = 0

    def _take(self) -> int:
        """Pop the head of the free queue; a cached block loses its hash (eviction)."""
        b = self.free_queue.popleft()
        if b in self.hash_of:
            h = self.hash_of.pop(b)
            if self.by_hash.get(h) == b:
                del self.by_hash[h]
            self.evictions += 1
        return b

    # -- a2: alloc / incref / free ------------------------------------------------
    def alloc(self, n: int) -> List[int]:
        """Take n blocks from the head of the free queue, each with refcount 1."""
        if n < 0:
            raise PoolError(INVALID_ARG, "negative count")
        if n > len(self.free_queue):
            raise PoolError(OUT_OF_BLOCKS, f"want {n}, have {len(self.free_queue)}")
        ids = [self._take() for _ in range(n)]
        for b in ids:
            self.refcount[b] = 1
        return ids

    def _check_ids(self, ids: Sequence[int]) -> None:
        for b in ids:
            if not (0 <= b < self.num_blocks):
                raise PoolError(BAD_BLOCK, f"block {b} out of range")

    def incref(self, ids: Sequence[int]) -> None:
        """One more reference to each listed block (sharing); free blocks are refused."""
        ids = [int(b) for b in ids]
        self._check_ids(ids)
        for b in ids:
            if self.refcount[b] == 0:
                raise PoolError(REFCOUNT, f"block {b} is free")
        for b in ids:
            self.refcount[b] += 1

    def free(self, ids: Sequence[int]) -> None:
        """Drop one reference per listed block; a block reaching 0 goes to the queue tail."""
        ids = [int(b) for b in ids]
        self._check_ids(ids)
        want: dict = {}
        for b in ids:
            want[b] = want.get(b, 0) + 1
        for b, k in want.items():
            if self.refcount[b] < k:
                raise PoolError(REFCOUNT, f"block {b} has refcount {self.refcount[b]} < {k}")
        for b in ids:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free_queue.append(b)

    # -- a3: append-slot + COW ------------------------------------------------------
    def prepare_append(self, tables: List[List[int]], lens: List[int], num_new: Sequence[int],
                       block_size: int, max_blocks: int):
        """Give slots to the next ``num_new[s]`` tokens of every sequence s.

        ``tables[s]`` (length ``max_blocks``, -1 = empty) and ``lens[s]`` are
        updated in place. Returns ``(slot_mapping, copy_pairs)``: one slot per new
        token in (sequence, token) order, and the (src, dst) blocks to copy before
        the new tokens are written. All-or-nothing: on failure nothing changes.
        """
        if block_size <= 0 or max_blocks <= 0 or len(tables) != len(lens) or len(num_new) != len(lens):
            raise PoolError(INVALID_ARG, "bad shapes")
        saved = (copy.deepcopy(tables), list(lens), deque(self.free_queue), list(self.refcount), self.cow_copies,
                 dict(self.hash_of), dict(self.by_hash), self.evictions)
        try:
            slots: List[int] = []
            pairs: List[tuple] = []
            for s in range(len(lens)):
                if num_new[s] < 0:
                    raise PoolError(INVALID_ARG, "negative token count")
                for _ in range(int(num_new[s])):
                    p = lens[s]
                    logical, offset = divmod(p, block_size)
                    if logical >= max_blocks:
                        raise PoolError(INVALID_ARG, f"sequence {s} needs more than {max_blocks} blocks")
                    if offset == 0:
                        tables[s][logical] = self.alloc(1)[0]
                    else:
                        cur = tables[s][logical]
                        if not (0 <= cur < self.num_blocks) or self.refcount[cur] == 0:
                            raise PoolError(BAD_BLOCK, f"sequence {s} logical block {logical} = {cur}")
                        if self.refcount[cur] > 1:
                            dst = self.alloc(1)[0]
                            pairs.append((cur, dst))
                            self.refcount[cur] -= 1
                            self.cow_copies += 1
                            tables[s][logical] = dst
                    slots.append(tables[s][logical] * block_size + offset)
                    lens[s] = p + 1
            return slots, pairs
        except PoolError:
            tables[:] = saved[0]
            lens[:] = saved[1]
            self.free_queue = saved[2]
            self.refcount = saved[3]
            self.cow_copies = saved[4]
            self.hash_of, self.by_hash, self.evictions = saved[5], saved[6], saved[7]
            raise

    # -- prefix cache ---------------------------------------------------------------
    def prefix_lookup(self, hashes: Sequence[int]) -> List[int]:
        """Blocks of the leading run of cached hashes; each gets one more reference."""
        ids: List[int] = []
        for h in hashes:
            b = self.by_hash.get(int(h))
            if b is None:
                break
            if self.refcount[b] == 0:
                self.free_queue.remove(b)      # a cached free block is revived
            self.refcount[b] += 1
            ids.append(b)
        self.prefix_hits += len(ids)
        self.prefix_misses += len(hashes) - len(ids)
        return ids

    def prefix_register(self, hashes: Sequence[int], ids: Sequence[int]) -> None:
        """Record full, written blocks under their hashes (first holder of a hash keeps it)."""
        ids = [int(b) for b in ids]
        self._check_ids(ids)
        for b in ids:
            if self.refcount[b] == 0:
                raise PoolError(REFCOUNT, f"block {b} is free")
        for h, b in zip((int(x) for x in hashes), ids):
            if b in self.hash_of:
                if self.hash_of[b] == h:
                    continue
                old = self.hash_of.pop(b)
                if self.by_hash.get(old) == b:
                    del self.by_hash[old]
            if h in self.by_hash:
                continue
            self.by_hash[h] = b
            self.hash_of[b] = h

    # -- bookkeeping ------------------------------------------------------------------
    def stats(self) -> PoolStats:
        used = sum(1 for r in self.refcount if r > 0)
        return PoolStats(
            free_blocks=len(self.free_queue),
            used_blocks=used,
            shared_blocks=sum(1 for r in self.refcount if r > 1),
            max_refcount=max(self.refcount) if self.refcount else 0,
            cow_copies=self.cow_copies,
            cached_blocks=len(self.hash_of),
            cached_free_blocks=sum(1 for b in self.hash_of if self.refcount[b] == 0),
            prefix_hits=self.prefix_hits,
            prefix_misses=self.prefix_misses,
            evictions=self.evictions,
        )

    def validate(self) -> None:
        """Free queue holds exactly the blocks with refcount 0, each once."""
        q = list(self.free_queue)
        if len(set(q)) != len(q):
            raise PoolError(REFCOUNT, "duplicate in free queue")
        zero = {b for b, r in enumerate(self.refcount) if r == 0}
        if set(q) != zero:
            raise PoolError(REFCOUNT, "free queue and zero refcounts disagree")
        if any(r < 0 for r in self.refcount):
            raise PoolError(REFCOUNT, "negative refcount")
        for b, h in self.hash_of.items():
            if self.by_hash.get(h) != b:
                raise PoolError(REFCOUNT, f"cached block {b} missing from the map")
        for h, b in self.by_hash.items():
            if self.hash_of.get(b) != h:
                raise PoolError(REFCOUNT, f"map entry {h:#x} without its block")


def admit(pool: RefPool, num_tokens: int, block_size: int, max_blocks: int) -> List[int]:
    """Table row of a new sequence of ``num_tokens`` tokens (all blocks fresh)."""
    need = -(-num_tokens // block_size)
    if need > max_blocks:
        raise PoolError(INVALID_ARG, "table too small")
    ids = pool.alloc(need)
    return ids + [-1] * (max_blocks - need)


def fork(pool: RefPool, table_row: Sequence[int], num_tokens: int, block_size: int) -> List[int]:
    """Table row of a sequence sharing all blocks of ``table_row`` (refcount +1 each)."""
    need = -(-num_tokens // block_size)
    pool.incref(list(table_row[:need]))
    return list(table_row)
