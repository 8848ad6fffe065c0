"""Pins of the swap oracle (``OracleEngine.swap_out`` / ``swap_in``), on the CPU.

Swap is preemption by copying (icman.com.cn/news/78786 §4.2): a request's KV
blocks leave the pool for host memory and their blocks go back to the free
queue; later the request is given fresh blocks and its KV is written back into
them. What fixes the result independently of the oracle's own code:

* every row of the swapped sequences (K and V codes, and for an E4M3 cache the
  K and V row scales, in every layer) reads back bit for bit through the new
  table, after other requests have taken every free block and written junk;
* the attention of every sequence (swapped or not) is bit-identical to its
  value before the swap (same values gathered in the same order);
* the allocator's state follows the FIFO / refcount rules by hand: swap-out
  pushes exactly the blocks whose refcount reaches 0 to the tail in table
  order (a block still shared with another sequence stays), the churn takes the
  whole queue from the head, and swap-in takes its blocks from the head with
  refcount 1 (hnwysp.cn/news/103996 §3.3, §3.4);
* a planted mistake (scales not saved, data written to the old ids, K and V
  swapped, blocks not released, blocks written back in the wrong order) makes
  the check fail.
"""
import numpy as np
import pytest

import workloads as wl
from oracle import fp8
from oracle import ref_attn as rf
from oracle.driver import OracleEngine

SWAPPED = (1, 3)


def _oracle(w, cls=OracleEngine):
    if w.kv_dtype == "e4m3":
        return cls(w, wl.pool_codes_e4m3(w, 0), wl.pool_codes_e4m3(w, 1), wl.pool_scales(w, 0),
                   wl.pool_scales(w, 1))
    return cls(w, wl.pool_values(w, 0), wl.pool_values(w, 1))


def _attention(ora, q):
    """Every layer's attention on the oracle's current state, float64 [L, S, H, D]."""
    w = ora.w
    tab = ora.tables_array()
    out = []
    for layer in range(w.num_layers):
        if ora.q8:
            out.append(fp8.decode_attention(q[layer], ora.k_pool[layer], ora.v_pool[layer], ora.k_scale[layer],
                                            ora.v_scale[layer], tab, ora.lens, w.block_size))
        else:
            out.append(rf.decode_attention(q[layer], ora.k_pool[layer], ora.v_pool[layer], tab, ora.lens,
                                           w.block_size, w.layout))
    return np.stack(out)


def _rows(ora, ids):
    """The test's own read of blocks ``ids`` in every array: [K, V(, K scale, V scale)][L, n, ...]."""
    arrs = [ora.k_pool, ora.v_pool] + ([ora.k_scale, ora.v_scale] if ora.q8 else [])
    return [a[:, list(ids)].copy() for a in arrs]


def check_swap(w, cls=OracleEngine) -> bool:
    """True when swap-out / churn / swap-in of two sequences behaves as the rules fix it."""
    ora = _oracle(w, cls)
    ora.run_script()
    B = w.block_size
    q = np.stack([wl.query_values(w, 0, l) for l in range(w.num_layers)])
    att0 = _attention(ora, q)
    nblk = {s: -(-ora.lens[s] // B) for s in SWAPPED}
    old_ids = {s: list(ora.tables[s][:nblk[s]]) for s in SWAPPED}
    rows0 = {s: _rows(ora, old_ids[s]) for s in SWAPPED}
    lens0 = list(ora.lens)
    ref0 = {b: ora.pool.refcount[b] for s in SWAPPED for b in old_ids[s]}
    queue0 = list(ora.pool.free_queue)

    # ---- swap out: refcounts drop by one per table reference; blocks reaching 0 go to the tail
    saved = {}
    expect_queue = list(queue0)
    refs = dict(ref0)
    for s in SWAPPED:
        saved[s] = ora.swap_out(s)
        for b in old_ids[s]:
            refs[b] -= 1
            if refs[b] == 0:
                expect_queue.append(b)
    if list(ora.pool.free_queue) != expect_queue:
        return False
    if any(ora.pool.refcount[b] != refs[b] for b in refs):
        return False
    if any(any(x != -1 for x in ora.tables[s]) for s in SWAPPED) or list(ora.lens) != lens0:
        return False

    # ---- churn: another request takes the whole queue (head first), writes junk and leaves
    junk = ora.pool.alloc(len(expect_queue))
    if junk != expect_queue:
        return False
    for a in [ora.k_pool, ora.v_pool] + ([ora.k_scale, ora.v_scale] if ora.q8 else []):
        blk = a[:, junk]
        a[:, junk] = np.frombuffer(b"\x5a" * blk.nbytes, dtype=a.dtype).reshape(blk.shape)
    ora.pool.free(junk)
    if list(ora.pool.free_queue) != junk:
        return False

    # ---- swap in: fresh blocks from the head of the queue, refcount 1, data back bit for bit
    head = 0
    for s in SWAPPED:
        ora.swap_in(s, saved[s])
        want = junk[head:head + nblk[s]]
        head += nblk[s]
        if list(ora.tables[s][:nblk[s]]) != want or any(x != -1 for x in ora.tables[s][nblk[s]:]):
            return False
        if any(ora.pool.refcount[b] != 1 for b in want):
            return False
        got = _rows(ora, want)
        for a, b in zip(got, rows0[s]):
            if not np.array_equal(a.view(np.uint8), b.view(np.uint8)):
                return False
    if list(ora.pool.free_queue) != junk[head:]:
        return False
    ora.pool.validate()
    # every sequence attends to exactly what it did before the swap
    return np.array_equal(_attention(ora, q), att0)


def _workloads():
    # the forked-prompt workload: the swapped sequences share the prompt's full blocks with
    # the others (those stay in the pool) and own their private suffix blocks (those are freed)
    # (20 decode steps of headroom size the pool so that swap-in finds enough free blocks)
    return [wl.make_workload(3, num_layers=2, num_seqs=5, len_scale=0.1, decode_steps=20),
            wl.make_workload(3, num_layers=2, num_seqs=5, len_scale=0.1, decode_steps=20, kv_dtype="e4m3"),
            wl.make_workload(2, num_layers=2, num_seqs=5, len_scale=0.05, decode_steps=2, layout="NHD")]


@pytest.mark.parametrize("i", [0, 1, 2], ids=["f16-prefix", "e4m3-prefix", "f16-7b-nhd"])
def test_swap_oracle_round_trip(i):
    w = _workloads()[i]
    assert check_swap(w)


def test_swapped_sequence_shares_prefix_blocks():
    """The case really exercises shared blocks: some of a swapped sequence's blocks stay in the pool."""
    w = _workloads()[0]
    ora = _oracle(w)
    ora.run_script()
    ids = ora.tables[SWAPPED[0]][:-(-ora.lens[SWAPPED[0]] // w.block_size)]
    assert any(ora.pool.refcount[b] > 1 for b in ids) and any(ora.pool.refcount[b] == 1 for b in ids)


# --------------------------------------------------------------------------- planted mistakes

class _Mutant(OracleEngine):
    kind = "none"

    def swap_out(self, s):
        B = self.w.block_size
        n = -(-self.lens[s] // B)
        ids = self.tables[s][:n]
        arrs = self._arrays()
        if self.kind == "scales_not_saved":
            arrs = arrs[:2]
        saved = [a[:, ids].copy() for a in arrs]
        if self.kind == "k_v_swapped":
            saved[0], saved[1] = saved[1], saved[0]
        if self.kind != "blocks_not_released":
            self.pool.free(ids)
        self.tables[s] = [-1] * self.w.max_blocks
        return (saved, list(ids))

    def swap_in(self, s, saved):
        saved, old = saved
        n = saved[0].shape[1]
        ids = self.pool.alloc(n)
        self.tables[s] = ids + [-1] * (self.w.max_blocks - n)
        dst = old if self.kind == "written_to_old_ids" else ids
        for a, v in zip(self._arrays(), saved):
            a[:, dst] = v[:, ::-1] if self.kind == "reversed_order" else v


def _mutant(kind):
    return type(f"Mutant_{kind}", (_Mutant,), {"kind": kind})


@pytest.mark.parametrize("kind", ["scales_not_saved", "k_v_swapped", "blocks_not_released", "written_to_old_ids",
                                  "reversed_order"])
def test_planted_swap_mistake_is_caught(kind):
    ws = _workloads()
    # the scale slip only exists on an E4M3 cache
    cases = [ws[1]] if kind == "scales_not_saved" else ws
    results = []
    for w in cases:
        try:
            results.append(check_swap(w, _mutant(kind)))
        except Exception:
            results.append(False)
    assert not all(results), f"planted mistake {kind} not caught"


def test_unmutated_copy_passes():
    for w in _workloads():
        assert check_swap(w, _mutant("none"))
