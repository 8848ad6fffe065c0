"""Pins of the allocator oracle (oracle/ref_alloc.py).

Hand-worked scenarios follow the pages' rules (head-of-queue allocation, tail
return, refcount, copy-on-write at the fork point); invariants are checked over
seeded random and exhaustively enumerated operation sequences.
"""
import itertools
import random

import numpy as np
import pytest

from oracle import ref_alloc as ra
import workloads


def test_fifo_refcount_worked_example():
    p = ra.RefPool(4, [2, 0, 3, 1])
    assert p.alloc(2) == [2, 0]
    assert list(p.free_queue) == [3, 1]
    p.incref([0])
    assert p.refcount == [2, 0, 1, 0]
    p.free([2])
    assert list(p.free_queue) == [3, 1, 2]
    p.free([0])
    assert p.refcount[0] == 1 and list(p.free_queue) == [3, 1, 2]
    assert p.alloc(3) == [3, 1, 2]
    with pytest.raises(ra.PoolError) as e:
        p.alloc(1)
    assert e.value.code == ra.OUT_OF_BLOCKS
    assert p.refcount == [1, 1, 1, 1] and list(p.free_queue) == []
    p.free([0, 3])
    assert list(p.free_queue) == [0, 3]
    with pytest.raises(ra.PoolError) as e:
        p.free([0])
    assert e.value.code == ra.REFCOUNT
    with pytest.raises(ra.PoolError) as e:
        p.incref([3])            # a free block cannot be shared
    assert e.value.code == ra.REFCOUNT
    with pytest.raises(ra.PoolError) as e:
        p.free([4])
    assert e.value.code == ra.BAD_BLOCK
    p.validate()


def test_free_is_all_or_nothing():
    p = ra.RefPool(3)
    ids = p.alloc(2)
    with pytest.raises(ra.PoolError):
        p.free([ids[0], ids[0]])     # refcount 1 cannot be dropped twice
    assert p.refcount[ids[0]] == 1 and list(p.free_queue) == [2]


def test_cow_worked_example():
    B = 4
    p = ra.RefPool(8)
    t0 = ra.admit(p, 5, B, 4)          # blocks 0, 1
    assert t0 == [0, 1, -1, -1]
    t1 = ra.fork(p, t0, 5, B)
    assert p.refcount[:2] == [2, 2]
    tables, lens = [t0, t1], [5, 5]
    slots, pairs = p.prepare_append(tables, lens, [1, 1], B, 4)
    # seq 0 writes into shared block 1 -> copy to fresh block 2; seq 1 then owns block 1 alone
    assert pairs == [(1, 2)]
    assert slots == [2 * 4 + 1, 1 * 4 + 1]
    assert tables == [[0, 2, -1, -1], [0, 1, -1, -1]]
    assert lens == [6, 6]
    assert p.refcount[:3] == [2, 1, 1]
    slots, pairs = p.prepare_append(tables, lens, [3, 0], B, 4)
    assert pairs == [] and slots == [10, 11, 3 * 4 + 0]
    assert tables[0] == [0, 2, 3, -1] and lens == [9, 6]
    assert p.cow_copies == 1
    p.validate()


def test_prepare_append_rolls_back_on_failure():
    B = 2
    p = ra.RefPool(3)
    t0 = ra.admit(p, 2, B, 3)
    t1 = ra.fork(p, t0, 2, B)
    tables, lens = [t0, t1], [2, 2]
    before = (list(map(list, tables)), list(lens), list(p.free_queue), list(p.refcount))
    with pytest.raises(ra.PoolError) as e:
        p.prepare_append(tables, lens, [3, 3], B, 3)   # needs 4 blocks, 2 are free
    assert e.value.code == ra.OUT_OF_BLOCKS
    assert (tables, lens, list(p.free_queue), list(p.refcount)) == before
    with pytest.raises(ra.PoolError) as e:
        p.prepare_append(tables, lens, [5, 0], B, 3)   # table too short
    assert e.value.code in (ra.INVALID_ARG, ra.OUT_OF_BLOCKS)
    assert (tables, lens, list(p.free_queue), list(p.refcount)) == before


def test_tiny_workload_tables_and_slots():
    w = workloads.make_workload(1)
    perm = [int(x) for x in w.free_order]
    p = ra.RefPool(w.num_blocks, perm)
    tables = [ra.admit(p, t, w.block_size, w.max_blocks) for t in w.context_lens]
    # 17, 33, 50, 64 tokens take 2, 3, 4, 4 blocks: consecutive runs of the queue
    assert [t[:n] for t, n in zip(tables, [2, 3, 4, 4])] == [perm[0:2], perm[2:5], perm[5:9], perm[9:13]]
    lens = [int(x) for x in w.context_lens]
    slots, pairs = p.prepare_append(tables, lens, [1, 1, 1, 1], w.block_size, w.max_blocks)
    assert pairs == []
    assert slots == [perm[1] * 16 + 1, perm[4] * 16 + 1, perm[8] * 16 + 2, perm[13] * 16 + 0]
    assert lens == [18, 34, 51, 65]


def test_prefix_workload_sharing_counts():
    """64 sequences forked from a 520-token prompt: 33 shared blocks, 63 COW copies."""
    w = workloads.make_workload(3, num_layers=1)
    p = ra.RefPool(w.num_blocks, [int(x) for x in w.free_order])
    B = w.block_size
    tables, lens = {}, {}
    for op in w.script:
        if op[0] == "admit":
            tables[op[1]] = ra.admit(p, op[2], B, w.max_blocks)
            lens[op[1]] = op[2]
        elif op[0] == "fork":
            tables[op[2]] = ra.fork(p, tables[op[1]], lens[op[1]], B)
            lens[op[2]] = lens[op[1]]
    S = w.num_seqs
    assert p.stats().max_refcount == S and p.stats().used_blocks == 33
    tl = [tables[s] for s in range(S)]
    ll = [lens[s] for s in range(S)]
    suffix = w.script[-1][1]
    slots, pairs = p.prepare_append(tl, ll, suffix, B, w.max_blocks)
    assert len(pairs) == S - 1 and all(src == tl[-1][32] for src, _ in pairs)
    st = p.stats()
    # memory is shared prefix + one copy per forked writer + private growth
    private = sum(-(-(520 + int(x)) // B) - 33 for x in suffix)
    assert st.used_blocks == 33 + (S - 1) + private
    assert st.cow_copies == S - 1
    assert st.shared_blocks == 32
    unshared = sum(-(-(520 + int(x)) // B) for x in suffix)
    assert st.used_blocks < unshared
    assert len(slots) == sum(suffix) and len(set(slots)) == len(slots)


def _check_invariants(p: ra.RefPool, seqs: dict, B: int):
    p.validate()
    st = p.stats()
    assert st.free_blocks + st.used_blocks == p.num_blocks
    refs = [0] * p.num_blocks
    for table, T in seqs.values():
        for b in table[: -(-T // B)]:
            refs[b] += 1
    assert refs == p.refcount


def _random_ops(seed: int, N: int, B: int, n_ops: int):
    rng = random.Random(seed)
    p = ra.RefPool(N, rng.sample(range(N), N))
    seqs = {}
    nxt = 0
    maxb = 8
    for _ in range(n_ops):
        op = rng.choice(["admit", "fork", "free", "append"])
        try:
            if op == "admit":
                T = rng.randint(1, 3 * B)
                seqs[nxt] = (ra.admit(p, T, B, maxb), T)
                nxt += 1
            elif op == "fork" and seqs:
                k = rng.choice(sorted(seqs))
                t, T = seqs[k]
                seqs[nxt] = (ra.fork(p, t, T, B), T)
                nxt += 1
            elif op == "free" and seqs:
                k = rng.choice(sorted(seqs))
                t, T = seqs.pop(k)
                p.free(t[: -(-T // B)])
            elif op == "append" and seqs:
                keys = sorted(seqs)
                tables = [list(seqs[k][0]) for k in keys]
                lens = [seqs[k][1] for k in keys]
                counts = [rng.randint(0, 3) for _ in keys]
                slots, pairs = p.prepare_append(tables, lens, counts, B, maxb)
                assert len(slots) == sum(counts)
                for k, t, T in zip(keys, tables, lens):
                    seqs[k] = (t, T)
        except ra.PoolError as e:
            assert e.code in (ra.OUT_OF_BLOCKS, ra.INVALID_ARG)
        _check_invariants(p, seqs, B)
    for k in sorted(seqs):
        t, T = seqs.pop(k)
        p.free(t[: -(-T // B)])
    assert all(r == 0 for r in p.refcount)
    assert sorted(p.free_queue) == list(range(N))


@pytest.mark.parametrize("seed", range(20))
def test_invariants_random_ops(seed):
    _random_ops(seed, N=12, B=4, n_ops=200)


def test_exhaustive_short_sequences():
    """Every sequence of up to 5 operations on a 3-block pool keeps the invariants."""
    B = 2
    ops = ["admit1", "admit3", "fork", "free", "append1", "append2"]
    count = 0
    for n in range(1, 6):
        for seq in itertools.product(ops, repeat=n):
            p = ra.RefPool(3)
            seqs = {}
            nxt = 0
            for op in seq:
                try:
                    if op.startswith("admit"):
                        T = int(op[-1])
                        seqs[nxt] = (ra.admit(p, T, B, 4), T)
                        nxt += 1
                    elif op == "fork" and seqs:
                        t, T = seqs[max(seqs)]
                        seqs[nxt] = (ra.fork(p, t, T, B), T)
                        nxt += 1
                    elif op == "free" and seqs:
                        t, T = seqs.pop(min(seqs))
                        p.free(t[: -(-T // B)])
                    elif op.startswith("append") and seqs:
                        keys = sorted(seqs)
                        tables = [list(seqs[k][0]) for k in keys]
                        lens = [seqs[k][1] for k in keys]
                        before_q = list(p.free_queue)
                        try:
                            p.prepare_append(tables, lens, [int(op[-1])] * len(keys), B, 4)
                        except ra.PoolError:
                            assert list(p.free_queue) == before_q
                            raise
                        for k, t, T in zip(keys, tables, lens):
                            seqs[k] = (t, T)
                except ra.PoolError:
                    pass
                _check_invariants(p, seqs, B)
            count += 1
    assert count == sum(len(ops) ** n for n in range(1, 6))


def test_cow_keeps_other_readers_data_model():
    """After a COW, the reader that kept the old block still maps the old block."""
    B = 4
    p = ra.RefPool(6)
    t0 = ra.admit(p, 6, B, 3)
    t1 = ra.fork(p, t0, 6, B)
    t2 = ra.fork(p, t0, 6, B)
    tables, lens = [t0, t1, t2], [6, 6, 6]
    _, pairs = p.prepare_append(tables, lens, [1, 1, 1], B, 3)
    # seqs 0 and 1 copy (refcount 3 then 2); seq 2 writes in place
    assert [d for _, d in pairs] == [tables[0][1], tables[1][1]]
    assert tables[2][1] == 1
    assert tables[0][0] == tables[1][0] == tables[2][0] == 0
    assert p.refcount[0] == 3 and p.refcount[1] == 1


def test_config_free_orders_are_permutations():
    for i in range(1, 6):
        w = workloads.make_workload(i)
        assert sorted(w.free_order.tolist()) == list(range(w.num_blocks))
        assert np.any(w.free_order != np.arange(w.num_blocks))


# --------------------------------------------------------------------------- planted mistakes
# The worked examples above as checks of a given pool class, and copies of the oracle's
# pool with one plausible slip each: every slip makes at least one check fail.

def _ok(fn):
    try:
        return bool(fn())
    except Exception:
        return False


def _check_fifo(P):
    p = P(4, [2, 0, 3, 1])
    if p.alloc(2) != [2, 0]:
        return False
    p.incref([0])
    p.free([2])
    p.free([0])
    if list(p.free_queue) != [3, 1, 2] or p.alloc(3) != [3, 1, 2]:
        return False
    try:
        p.alloc(1)
        return False
    except ra.PoolError:
        pass
    p.free([0, 3])
    return list(p.free_queue) == [0, 3] and p.refcount == [0, 1, 1, 0]


def _check_cow(P):
    B, p = 4, P(8)
    t0 = ra.admit(p, 5, B, 4)
    t1 = ra.fork(p, t0, 5, B)
    tables, lens = [t0, t1], [5, 5]
    slots, pairs = p.prepare_append(tables, lens, [1, 1], B, 4)
    return (pairs == [(1, 2)] and slots == [9, 5] and tables == [[0, 2, -1, -1], [0, 1, -1, -1]]
            and p.refcount[:3] == [2, 1, 1] and p.cow_copies == 1)


def _check_rollback(P):
    B, p = 2, P(3)
    t0 = ra.admit(p, 2, B, 3)
    t1 = ra.fork(p, t0, 2, B)
    tables, lens = [t0, t1], [2, 2]
    before = (list(map(list, tables)), list(lens), list(p.free_queue), list(p.refcount))
    try:
        p.prepare_append(tables, lens, [3, 3], B, 3)
        return False
    except ra.PoolError:
        pass
    return (tables, lens, list(p.free_queue), list(p.refcount)) == before


def _check_tiny_slots(P):
    w = workloads.make_workload(1)
    perm = [int(x) for x in w.free_order]
    p = P(w.num_blocks, perm)
    tables = [ra.admit(p, t, w.block_size, w.max_blocks) for t in w.context_lens]
    lens = [int(x) for x in w.context_lens]
    slots, pairs = p.prepare_append(tables, lens, [1, 1, 1, 1], w.block_size, w.max_blocks)
    return pairs == [] and slots == [perm[1] * 16 + 1, perm[4] * 16 + 1, perm[8] * 16 + 2, perm[13] * 16 + 0]


def _check_alloc_all_or_nothing(P):
    p = P(3)
    p.alloc(2)
    try:
        p.alloc(2)
        return False
    except ra.PoolError:
        return list(p.free_queue) == [2] and p.refcount == [1, 1, 0]


class _LifoFree(ra.RefPool):
    def free(self, ids):
        for b in [int(x) for x in ids]:
            if self.refcount[b] < 1:
                raise ra.PoolError(ra.REFCOUNT, "free block")
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free_queue.appendleft(b)


class _PartialAlloc(ra.RefPool):
    def alloc(self, n):
        ids = []
        for _ in range(n):
            if not self.free_queue:
                raise ra.PoolError(ra.OUT_OF_BLOCKS, "empty")
            b = self._take()
            self.refcount[b] = 1
            ids.append(b)
        return ids


def _append_mutant(kind):
    class _P(ra.RefPool):
        def prepare_append(self, tables, lens, num_new, block_size, max_blocks):
            slots, pairs = [], []
            for s in range(len(lens)):
                for _ in range(int(num_new[s])):
                    p = lens[s]
                    logical, offset = divmod(p, block_size)
                    if logical >= max_blocks:
                        raise ra.PoolError(ra.INVALID_ARG, "table too short")
                    if offset == 0:
                        tables[s][logical] = self.alloc(1)[0]
                    else:
                        cur = tables[s][logical]
                        if self.refcount[cur] > 1 and kind != "no_cow":
                            dst = self.alloc(1)[0]
                            pairs.append((cur, dst))
                            if kind != "cow_no_decref":
                                self.refcount[cur] -= 1
                            self.cow_copies += 1
                            tables[s][logical] = dst
                    blk = logical if kind == "logical_slot" else tables[s][logical]
                    slots.append(blk * block_size + offset)
                    lens[s] = p + 1
            return slots, pairs       # kind "no_rollback" too: nothing restored on failure
    return _P


_MUTANTS = {"lifo_free": _LifoFree, "partial_alloc": _PartialAlloc, "no_cow": _append_mutant("no_cow"),
            "cow_no_decref": _append_mutant("cow_no_decref"), "logical_slot": _append_mutant("logical_slot"),
            "no_rollback": _append_mutant("no_rollback")}
_CHECKS = (_check_fifo, _check_cow, _check_rollback, _check_tiny_slots, _check_alloc_all_or_nothing)


@pytest.mark.parametrize("kind", sorted(_MUTANTS))
def test_planted_allocator_mistake_is_caught(kind):
    P = _MUTANTS[kind]
    assert not all(_ok(lambda c=c: c(P)) for c in _CHECKS), kind


def test_oracle_pool_passes_the_checks():
    assert all(_ok(lambda c=c: c(ra.RefPool)) for c in _CHECKS)
