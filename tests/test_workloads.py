"""The seeded input recipe of the five workloads (shapes, seeds, length distributions, pool
sizing) and its determinism: the generators both sides draw from give the same inputs on
every call. The module holds no arithmetic of the method; these pins keep the recipe the
design notes state."""
import math

import numpy as np
import pytest

import workloads as wl

SHAPES = {  # index: (name, L, H, D, B, S)
    1: ("tiny", 1, 4, 64, 16, 4),
    2: ("7b", 32, 32, 128, 16, 32),
    3: ("prefix", 32, 32, 128, 16, 64),
    4: ("13b", 40, 40, 128, 32, 128),
    5: ("long", 32, 32, 128, 256, 16),
}


@pytest.mark.parametrize("index", sorted(SHAPES))
def test_shapes_and_seeds(index):
    w = wl.make_workload(index)
    name, L, H, D, B, S = SHAPES[index]
    assert (w.name, w.num_layers, w.num_heads, w.head_dim, w.block_size, w.num_seqs) == (name, L, H, D, B, S)
    assert w.seed == 1000 + index
    assert sorted(int(x) for x in w.free_order) == list(range(w.num_blocks))


def test_length_distributions():
    assert [int(t) for t in wl.make_workload(1).context_lens] == [17, 33, 50, 64]
    l2 = np.asarray(wl.make_workload(2).context_lens)
    assert l2.min() >= 256 and l2.max() <= 2048
    w3 = wl.make_workload(3)
    l3 = np.asarray(w3.context_lens)
    assert l3.min() >= 520 + 64 and l3.max() <= 520 + 512
    l4 = np.asarray(wl.make_workload(4).context_lens)
    assert l4.min() >= 16 and l4.max() <= 4096 and 200 <= np.median(l4) <= 450   # lognormal, median 300
    l5 = np.asarray(wl.make_workload(5).context_lens)
    assert l5.min() >= 4096 and l5.max() <= 16384


def test_pool_sizing():
    # the 7B pool: 1.3x the blocks its batch needs
    w = wl.make_workload(2)
    need = sum(-(-int(t) // w.block_size) for t in w.context_lens)
    assert w.num_blocks >= math.ceil(1.3 * need)
    # the 13B pool is about 90 % occupied after the set-up's churn (replayed with the oracle
    # allocator: admissions, dummy allocations and frees)
    from oracle import ref_alloc as ra
    w4 = wl.make_workload(4)
    p = ra.RefPool(w4.num_blocks, [int(x) for x in w4.free_order])
    dummies = {}
    for op in w4.script:
        if op[0] == "admit":
            ra.admit(p, op[2], w4.block_size, w4.max_blocks)
        elif op[0] == "dummy_alloc":
            dummies[op[1]] = p.alloc(op[2])
        elif op[0] == "dummy_free":
            p.free(dummies.pop(op[1]))
    used = w4.num_blocks - len(p.free_queue)
    assert 0.85 <= used / w4.num_blocks <= 0.95


def test_sweep_block_sizes_keep_the_tokens():
    base = np.asarray(wl.make_workload(5).context_lens)
    for B in (8, 16, 32, 64, 512):
        w = wl.make_workload(5, block_size=B)
        assert w.block_size == B and np.array_equal(np.asarray(w.context_lens), base)


@pytest.mark.parametrize("index", [1, 2, 3])
def test_draws_are_deterministic(index):
    a, b = wl.make_workload(index, num_layers=1), wl.make_workload(index, num_layers=1)
    assert np.array_equal(np.asarray(a.context_lens), np.asarray(b.context_lens))
    assert np.array_equal(np.asarray(a.free_order), np.asarray(b.free_order))
    if index == 1:
        assert np.array_equal(wl.pool_values(a, 0), wl.pool_values(b, 0))
        assert np.array_equal(wl.query_values(a, 0, 0), wl.query_values(b, 0, 0))
        assert not np.array_equal(wl.query_values(a, 0, 0), wl.query_values(a, 1, 0))   # fresh per step
