"""CPU tests of the shared-prefix (cascade) planner, pkv_cascade_plan.

The plan only moves work between the prefix pass and the private pass, so it is
pinned by what must hold of any correct plan -- every member of a group holds
the same block ids over the group's prefix, the prefix is whole blocks inside
every member's context, groups are consecutive runs of at most 128 sequences --
plus hand-worked cases and the greedy rule's maximality.
"""
import numpy as np
import pytest

from paged_kv_cache_88_gb300 import binding as bd


def full_blocks(T, B, maxb):
    return max(0, min(T // B, maxb)) if T > 0 else 0


def check_plan(tab, lens, B, groups, begin, min_group=2, min_prefix=0):
    S, maxb = tab.shape
    min_blocks = max(1, -(-max(min_prefix, 0) // B))
    member = np.zeros(S, dtype=bool)
    for f, n, P, res in groups.tolist():
        assert res == 0
        assert min_group <= n <= bd.MAX_GROUP_SEQS
        assert P % B == 0 and P // B >= min_blocks
        nb = P // B
        for s in range(f, f + n):
            assert not member[s], "a sequence in two groups"
            member[s] = True
            assert begin[s] == P
            assert nb <= full_blocks(int(lens[s]), B, maxb), "prefix not wholly inside the context"
            assert (tab[s, :nb] == tab[f, :nb]).all() and (tab[f, :nb] >= 0).all()
    assert (begin[~member] == 0).all()
    # greedy maximality: the sequence right after a group could not have joined it
    for f, n, P, _ in groups.tolist():
        e = f + n
        if e < S and n < bd.MAX_GROUP_SEQS:
            nb = min(P // B, full_blocks(int(lens[e]), B, maxb))
            k = 0
            while k < nb and tab[f, k] >= 0 and tab[f, k] == tab[e, k]:
                k += 1
            assert k < min_blocks


def test_hand_worked_plan():
    tab = np.array([[5, 6, 7, -1], [5, 6, 8, -1], [5, 6, 7, 9], [1, 2, 3, 4]], dtype=np.int32)
    lens = np.array([40, 40, 60, 64], dtype=np.int32)
    groups, begin = bd.cascade_plan(tab, lens, 16)
    # sequences 0..2 share blocks 5, 6 (32 tokens); block 7 is shared by 0 and 2 only,
    # and sequence 0 holds just 2 full blocks anyway
    assert groups.tolist() == [[0, 3, 32, 0]]
    assert begin.tolist() == [32, 32, 32, 0]
    check_plan(tab, lens, 16, groups, begin)


def test_forked_prompt_plan():
    # a 520-token prompt forked into 64 requests, B = 16: 32 full shared blocks, the
    # partial 33rd copied per request (copy-on-write) before their suffixes
    B, S, maxb = 16, 64, 80
    rng = np.random.default_rng(3)
    tab = np.full((S, maxb), -1, dtype=np.int32)
    nxt = 32
    lens = np.zeros(S, dtype=np.int32)
    for s in range(S):
        T = 520 + int(rng.integers(64, 513))
        lens[s] = T
        nb = -(-T // B)
        tab[s, :32] = np.arange(32)
        tab[s, 32:nb] = np.arange(nxt, nxt + nb - 32)
        nxt += nb - 32
    groups, begin = bd.cascade_plan(tab, lens, B)
    assert groups.tolist() == [[0, 64, 512, 0]]
    assert (begin == 512).all()
    check_plan(tab, lens, B, groups, begin)


def test_group_size_cap_and_ragged_runs():
    B, S = 8, 300
    tab = np.tile(np.arange(10, dtype=np.int32), (S, 1))
    lens = np.full(S, 80, dtype=np.int32)
    groups, begin = bd.cascade_plan(tab, lens, B)
    assert groups.tolist() == [[0, 128, 80, 0], [128, 128, 80, 0], [256, 44, 80, 0]]
    check_plan(tab, lens, B, groups, begin)


def test_min_group_min_prefix_and_max_groups():
    B = 16
    # pairs sharing 2 blocks, a triple sharing 8 blocks
    tab = np.array([[0, 1, 2, 3, 4, 5, 6, 7],
                    [0, 1, 9, 9, 9, 9, 9, 9],
                    [20, 21, 22, 23, 24, 25, 26, 27],
                    [20, 21, 22, 23, 24, 25, 26, 27],
                    [20, 21, 22, 23, 24, 25, 26, 27]], dtype=np.int32)
    tab[1, 2:] = np.arange(40, 46)
    lens = np.full(5, 128, dtype=np.int32)
    g, b = bd.cascade_plan(tab, lens, B)
    assert g.tolist() == [[0, 2, 32, 0], [2, 3, 128, 0]]
    g, b = bd.cascade_plan(tab, lens, B, min_group=3)
    assert g.tolist() == [[2, 3, 128, 0]] and b.tolist() == [0, 0, 128, 128, 128]
    g, b = bd.cascade_plan(tab, lens, B, min_prefix_tokens=33)      # needs 3 blocks
    assert g.tolist() == [[2, 3, 128, 0]]
    g, b = bd.cascade_plan(tab, lens, B, max_groups=1)
    assert g.tolist() == [[0, 2, 32, 0]] and b.tolist() == [32, 32, 0, 0, 0]
    g, b = bd.cascade_plan(tab, lens, B, max_groups=0)
    assert len(g) == 0 and (b == 0).all()


def test_prefix_stops_at_partial_block_and_invalid_ids():
    B = 16
    tab = np.array([[3, 4, 5, -1], [3, 4, 5, -1], [-1, -1, -1, -1], [-1, -1, -1, -1]], dtype=np.int32)
    # block 5 is shared but sequence 1's context ends inside it
    lens = np.array([48, 40, 0, 0], dtype=np.int32)
    g, b = bd.cascade_plan(tab, lens, B)
    assert g.tolist() == [[0, 2, 32, 0]]
    # identical -1 entries are not a shared prefix
    assert b.tolist() == [32, 32, 0, 0]
    check_plan(tab, lens, B, g, b)


@pytest.mark.parametrize("seed", range(6))
def test_random_fork_trees(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([8, 16, 32, 64]))
    S, maxb = int(rng.integers(1, 200)), 24
    tab = np.full((S, maxb), -1, dtype=np.int32)
    lens = np.zeros(S, dtype=np.int32)
    nxt = 0
    for s in range(S):
        nb = int(rng.integers(0, maxb + 1))
        lens[s] = max(0, nb * B - int(rng.integers(0, B)))
        share = int(rng.integers(0, nb + 1)) if s and rng.random() < 0.7 else 0
        src = int(rng.integers(max(0, s - 3), s)) if share else 0
        share = min(share, int((tab[src] >= 0).sum()))
        tab[s, :share] = tab[src, :share]
        tab[s, share:nb] = np.arange(nxt, nxt + nb - share)
        nxt += nb - share
    for mg in (2, 3):
        for mp in (0, B, 3 * B):
            g, b = bd.cascade_plan(tab, lens, B, min_group=mg, min_prefix_tokens=mp)
            check_plan(tab, lens, B, g, b, mg, mp)


def test_bad_arguments():
    tab = np.zeros((2, 2), dtype=np.int32)
    lens = np.full(2, 32, dtype=np.int32)
    with pytest.raises(bd.PkvError) as e:
        bd.cascade_plan(tab, lens, 16, min_group=1)
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(bd.PkvError) as e:
        bd.cascade_plan(tab, lens, 12)
    assert e.value.code == "UNSUPPORTED"


def test_piece_buffer_size_and_splits():
    assert bd.prefix_pieces_bytes(64, 32, 128) == 64 * 32 * bd.MAX_PREFIX_SPLITS * 132 * 4
    assert bd.prefix_pieces_bytes(0, 32, 128) == 0
    for g, h, p in ((1, 32, 512), (4, 40, 4096), (1, 1, 100000), (0, 32, 512)):
        assert 1 <= bd.prefix_splits(g, h, p) <= bd.MAX_PREFIX_SPLITS
    assert bd.prefix_splits(1, 32, 128) == 1        # one key tile: one split
