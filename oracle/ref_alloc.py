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

Readings taken where the pages are silent (each is listed in the design doc):

* Allocation is all-or-nothing and a failed call changes nothing.
* COW fires iff the refcount of the block being written is > 1 at the moment of
  the write; sequences are processed in ascending index, tokens in order.
* A slot is ``physical_block * B + offset``; -1 in a table means "no block".
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


@dataclass
class PoolStats:
    free_blocks: int
    used_blocks: int
    shared_blocks: int
    max_refcount: int
    cow_copies: int


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

    # -- a2: alloc / incref / free ------------------------------------------------
    def alloc(self, n: int) -> List[int]:
        """Take n blocks from the head of the free queue, each with refcount 1."""
        if n < 0:
            raise PoolError(INVALID_ARG, "negative count")
        if n > len(self.free_queue):
            raise PoolError(OUT_OF_BLOCKS, f"want {n}, have {len(self.free_queue)}")
        ids = [self.free_queue.popleft() for _ in range(n)]
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
        saved = (copy.deepcopy(tables), list(lens), deque(self.free_queue), list(self.refcount), self.cow_copies)
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
            raise

    # -- bookkeeping ------------------------------------------------------------------
    def stats(self) -> PoolStats:
        used = sum(1 for r in self.refcount if r > 0)
        return PoolStats(
            free_blocks=len(self.free_queue),
            used_blocks=used,
            shared_blocks=sum(1 for r in self.refcount if r > 1),
            max_refcount=max(self.refcount) if self.refcount else 0,
            cow_copies=self.cow_copies,
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
