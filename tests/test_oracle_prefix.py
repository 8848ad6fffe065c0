"""Pins of the prefix-cache oracle (oracle/ref_alloc.py): the FNV-1a hash against its
published test vectors, the chaining of block hashes, and a hand-worked scenario of
sharing, reviving and evicting cached blocks."""
import json
import os
import random

import pytest

from oracle import ref_alloc as ra

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fnv1a64.json")))


def test_fnv1a64_published_vectors():
    assert ra.FNV64_OFFSET == int(GOLD["offset_basis"], 16)
    assert ra.FNV64_PRIME == int(GOLD["prime"], 16)
    for v in GOLD["vectors"]:
        assert ra.fnv1a64(v["input_ascii"].encode()) == int(v["hash"], 16), v


def test_block_hash_bytes_and_chaining():
    # the bytes hashed: parent (8 LE) then each token (4 LE, two's complement)
    assert ra.block_hash(0, []) == ra.fnv1a64(bytes(8))
    assert ra.block_hash(0x0102030405060708, [1, -1]) == ra.fnv1a64(
        bytes([8, 7, 6, 5, 4, 3, 2, 1, 1, 0, 0, 0, 0xFF, 0xFF, 0xFF, 0xFF]))
    rng = random.Random(0)
    toks = [rng.randrange(32000) for _ in range(64)]
    h = ra.prompt_block_hashes(toks, 16)
    assert len(h) == 4 and len(set(h)) == 4
    assert ra.prompt_block_hashes(toks + [5, 6, 7], 16) == h          # a partial block is not hashed
    other = list(toks)
    other[3] += 1                                                     # change one early token ...
    h2 = ra.prompt_block_hashes(other, 16)
    assert all(a != b for a, b in zip(h, h2))                         # ... every later hash changes
    other = list(toks)
    other[40] += 1
    h3 = ra.prompt_block_hashes(other, 16)
    assert h3[:2] == h[:2] and h3[2] != h[2] and h3[3] != h[3]


def test_share_revive_evict_worked_example():
    B = 2
    p = ra.RefPool(6)
    A = [1, 2, 3, 4, 5]
    hA = ra.prompt_block_hashes(A, B)
    assert p.prefix_lookup(hA) == []
    a_ids = p.alloc(3)
    assert a_ids == [0, 1, 2]
    p.prefix_register(hA, a_ids[:2])
    Bt = [1, 2, 3, 4, 9, 9]
    hB = ra.prompt_block_hashes(Bt, B)
    assert hB[:2] == hA
    assert p.prefix_lookup(hB) == [0, 1]                  # two shared blocks, then a miss
    assert p.refcount[:2] == [2, 2]
    b_ids = [0, 1] + p.alloc(1)
    assert b_ids == [0, 1, 3]
    p.prefix_register(hB[2:], b_ids[2:])
    p.free(a_ids)
    assert list(p.free_queue) == [4, 5, 2]
    p.free(b_ids)
    assert list(p.free_queue) == [4, 5, 2, 0, 1, 3]
    st = p.stats()
    assert (st.cached_blocks, st.cached_free_blocks) == (3, 3)
    assert p.prefix_lookup(hA) == [0, 1]                  # revived from the free queue
    assert list(p.free_queue) == [4, 5, 2, 3] and p.refcount[:2] == [1, 1]
    assert p.alloc(3) == [4, 5, 2] and p.stats().evictions == 0
    assert p.alloc(1) == [3] and p.stats().evictions == 1   # reusing a cached block evicts its hash
    assert p.prefix_lookup(hB) == [0, 1]
    st = p.stats()
    assert (st.prefix_hits, st.prefix_misses) == (6, 4)
    p.validate()


def test_register_rules():
    p = ra.RefPool(4)
    ids = p.alloc(2)
    p.prefix_register([11], [ids[0]])
    p.prefix_register([11], [ids[1]])                     # first holder keeps the hash
    assert p.by_hash[11] == ids[0] and ids[1] not in p.hash_of
    p.prefix_register([12], [ids[0]])                     # re-registered under a new hash
    assert 11 not in p.by_hash and p.by_hash[12] == ids[0]
    with pytest.raises(ra.PoolError):
        p.prefix_register([13], [3])                      # a free block
    p.validate()


@pytest.mark.parametrize("seed", range(8))
def test_prefix_invariants_random(seed):
    rng = random.Random(seed)
    B, N = 4, 24
    p = ra.RefPool(N, rng.sample(range(N), N))
    prefixes = [[rng.randrange(50) for _ in range(12)] for _ in range(3)]
    live = {}
    for step in range(150):
        if live and rng.random() < 0.35:
            k = rng.choice(sorted(live))
            p.free(live.pop(k))
        else:
            toks = rng.choice(prefixes)[: rng.randrange(4, 13)] + [rng.randrange(50) for _ in range(rng.randrange(5))]
            hs = ra.prompt_block_hashes(toks, B)
            hit = p.prefix_lookup(hs)
            need = -(-len(toks) // B) - len(hit)
            try:
                new = p.alloc(need)
            except ra.PoolError:
                p.free(hit)
                continue
            ids = hit + new
            p.prefix_register(hs[len(hit):], ids[len(hit):len(hs)])
            live[step] = ids
        p.validate()
        assert sum(p.refcount) == sum(len(v) for v in live.values())
    for k in list(live):
        p.free(live.pop(k))
    assert all(r == 0 for r in p.refcount) and sorted(p.free_queue) == list(range(N))


# --------------------------------------------------------------------------- planted mistakes
# The pins above as checks of a given (hash functions, pool class) and copies with one
# plausible slip each: every slip makes at least one check fail.

class _Impl:
    """The oracle's prefix-cache functions, with one slip when kind names one."""

    def __init__(self, kind):
        self.kind = kind
        impl = self

        class Pool(ra.RefPool):
            def prefix_lookup(self, hashes):
                ids = []
                for h in hashes:
                    b = self.by_hash.get(int(h))
                    if b is None:
                        if impl.kind == "lookup_past_miss":
                            continue
                        break
                    if self.refcount[b] == 0 and impl.kind != "revive_stays_queued":
                        self.free_queue.remove(b)
                    self.refcount[b] += 1
                    ids.append(b)
                self.prefix_hits += len(ids)
                self.prefix_misses += len(hashes) - len(ids)
                return ids
        self.Pool = Pool

    def fnv(self, data):
        h = ra.FNV64_OFFSET
        for byte in data:
            h = ((h * ra.FNV64_PRIME) ^ byte) & ra.MASK64 if self.kind == "fnv1_order" else \
                ((h ^ byte) * ra.FNV64_PRIME) & ra.MASK64
        return h

    def block_hash(self, parent, toks):
        if self.kind == "unchained":
            parent = 0
        return self.fnv(int(parent).to_bytes(8, "little") +
                        b"".join(int(t).to_bytes(4, "little", signed=True) for t in toks))

    def prompt_hashes(self, toks, B):
        out, parent = [], 0
        n = -(-len(toks) // B) if self.kind == "partial_block_hashed" else len(toks) // B
        for i in range(n):
            parent = self.block_hash(parent, toks[i * B:(i + 1) * B])
            out.append(parent)
        return out


def _check_vectors(m):
    return all(m.fnv(v["input_ascii"].encode()) == int(v["hash"], 16) for v in GOLD["vectors"])


def _check_chaining(m):
    rng = random.Random(0)
    toks = [rng.randrange(32000) for _ in range(64)]
    h = m.prompt_hashes(toks, 16)
    other = list(toks)
    other[3] += 1
    h2 = m.prompt_hashes(other, 16)
    return (len(h) == 4 and m.prompt_hashes(toks + [5, 6, 7], 16) == h and all(a != b for a, b in zip(h, h2)))


def _check_scenario(m):
    B, p = 2, m.Pool(6)
    hA = m.prompt_hashes([1, 2, 3, 4, 5], B)
    a_ids = p.alloc(3)
    p.prefix_register(hA, a_ids[:2])
    hB = m.prompt_hashes([1, 2, 3, 4, 9, 9], B)
    if p.prefix_lookup(hB) != [0, 1]:
        return False
    b_ids = [0, 1] + p.alloc(1)
    p.prefix_register(hB[2:], b_ids[2:])
    p.free(a_ids)
    p.free(b_ids)
    if p.prefix_lookup([hA[0], 12345, hA[1]]) != [0]:    # stops at the first miss
        return False
    p.validate()
    return list(p.free_queue) == [4, 5, 2, 1, 3]


@pytest.mark.parametrize("kind", ["fnv1_order", "unchained", "partial_block_hashed", "lookup_past_miss",
                                  "revive_stays_queued"])
def test_planted_prefix_cache_mistake_is_caught(kind):
    m = _Impl(kind)
    results = []
    for check in (_check_vectors, _check_chaining, _check_scenario):
        try:
            results.append(check(m))
        except Exception:
            results.append(False)
    assert not all(results), kind


def test_unmutated_prefix_cache_copy_passes():
    m = _Impl("none")
    assert _check_vectors(m) and _check_chaining(m) and _check_scenario(m)
