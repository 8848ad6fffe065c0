"""CPU tests of the C ABI: the library loads, exports every declared symbol, and its
host allocator reproduces the allocator oracle bit for bit (no GPU needed)."""
import ctypes
import os
import random
import re

import numpy as np
import pytest

import paged_kv_cache_88_gb300 as pkv
from paged_kv_cache_88_gb300 import binding as bd
from oracle import ref_alloc as ra
import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CODE = {ra.OUT_OF_BLOCKS: "OUT_OF_BLOCKS", ra.BAD_BLOCK: "BAD_BLOCK", ra.REFCOUNT: "REFCOUNT",
        ra.INVALID_ARG: "INVALID_ARG"}


def header_functions():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 19
    lib = pkv.lib()
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(bd.EXPORTED) == names


def test_library_exports_nothing_else():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", bd.LIB_PATH], capture_output=True, text=True).stdout
    syms = [l.split()[-1] for l in out.splitlines() if l.split() and l.split()[1] in "TtDdBbRr"]
    assert syms and all(s.startswith("pkv_") for s in syms), [s for s in syms if not s.startswith("pkv_")]


def test_version_and_error_text():
    assert pkv.lib().pkv_version() == 10000
    with pytest.raises(pkv.PkvError) as e:
        bd.Pool(1, 4, 12, 1, 64)          # block size 12 is not built
    assert e.value.code == "UNSUPPORTED"
    assert "block_size" in pkv.last_error()


def test_pool_create_rejects_bad_order():
    with pytest.raises(pkv.PkvError) as e:
        bd.Pool(1, 4, 16, 1, 64, initial_free_order=[0, 1, 1, 2])
    assert e.value.code == "INVALID_ARG"


def _pair(N, order=None):
    return bd.Pool(1, N, 8, 1, 64, initial_free_order=order), ra.RefPool(N, order)


def _same(c: bd.Pool, o: ra.RefPool):
    assert c.free_queue() == list(o.free_queue)
    assert [c.refcount(b) for b in range(o.num_blocks)] == o.refcount
    st = c.stats()
    os_ = o.stats()
    assert (st["free_blocks"], st["used_blocks"], st["shared_blocks"], st["max_refcount"], st["cow_copies"]) == \
        (os_.free_blocks, os_.used_blocks, os_.shared_blocks, os_.max_refcount, os_.cow_copies)
    c.validate()


def _both(fc, fo):
    """Run the same op on both; they must both succeed with equal results or fail with the same code."""
    try:
        ro = fo()
        eo = None
    except ra.PoolError as e:
        ro, eo = None, e.code
    try:
        rc = fc()
        ec = None
    except pkv.PkvError as e:
        rc, ec = None, e.code
    assert (ec is None) == (eo is None), (ec, eo)
    if eo is not None:
        assert ec == CODE[eo], (ec, eo)
    return rc, ro


@pytest.mark.parametrize("seed", range(12))
def test_allocator_matches_oracle_random_ops(seed):
    rng = random.Random(seed)
    N, B, maxb = 16, 8, 6
    order = rng.sample(range(N), N)
    c = bd.Pool(1, N, B, 1, 64, initial_free_order=order)
    o = ra.RefPool(N, order)
    seqs = {}
    nxt = 0
    for _ in range(300):
        op = rng.choice(["alloc", "free", "incref", "admit", "fork", "append", "dropseq", "badfree"])
        if op == "alloc":
            n = rng.randint(0, 5)
            rc, ro = _both(lambda: c.alloc(n), lambda: o.alloc(n))
            if ro is not None:
                assert rc == ro
                seqs[("raw", nxt)] = (ro + [-1] * (maxb - len(ro)), len(ro) * B)
                nxt += 1
        elif op == "admit":
            T = rng.randint(1, 3 * B)
            nb = -(-T // B)
            rc, ro = _both(lambda: c.alloc(nb), lambda: o.alloc(nb))
            if ro is not None:
                assert rc == ro
                seqs[nxt] = (ro + [-1] * (maxb - nb), T)
                nxt += 1
        elif op == "fork" and seqs:
            k = rng.choice(sorted(seqs, key=str))
            t, T = seqs[k]
            ids = t[: -(-T // B)]
            _both(lambda: c.incref(ids), lambda: o.incref(ids))
            seqs[nxt] = (list(t), T)
            nxt += 1
        elif op == "incref":
            ids = [rng.randint(-1, N) for _ in range(rng.randint(0, 3))]
            _both(lambda: c.incref(ids), lambda: o.incref(ids))
        elif op == "badfree":
            ids = [rng.randint(-1, N) for _ in range(rng.randint(0, 3))]
            _both(lambda: c.free(ids), lambda: o.free(ids))
        elif op == "dropseq" and seqs:
            k = rng.choice(sorted(seqs, key=str))
            t, T = seqs.pop(k)
            ids = t[: -(-T // B)]
            _both(lambda: c.free(ids), lambda: o.free(ids))
        elif op == "append" and seqs:
            keys = [k for k in sorted(seqs, key=str) if not (isinstance(k, tuple))]
            if not keys:
                continue
            counts = [rng.randint(0, 3) for _ in keys]
            tc = np.array([seqs[k][0] for k in keys], dtype=np.int32)
            lc = np.array([seqs[k][1] for k in keys], dtype=np.int32)
            to = [list(seqs[k][0]) for k in keys]
            lo = [seqs[k][1] for k in keys]
            rc, ro = _both(lambda: c.prepare_append(tc, lc, counts), lambda: o.prepare_append(to, lo, counts, B, maxb))
            assert tc.tolist() == to and lc.tolist() == lo
            if ro is not None:
                slots, pairs = rc
                assert slots.tolist() == ro[0]
                assert [tuple(p) for p in pairs.tolist()] == ro[1]
                for k, t, T in zip(keys, to, lo):
                    seqs[k] = (t, T)
        _same(c, o)


@pytest.mark.parametrize("index,mode", [(1, "fork"), (2, "fork"), (3, "fork"), (3, "hash"), (4, "fork"),
                                        (5, "fork")])
def test_workload_setup_tables_match_oracle(index, mode):
    """Every workload's set-up script (admit / fork / churn / COW writes / prefix-cache prompts) gives
    identical tables."""
    w = wl.make_workload(index, num_layers=1, prefix_mode=mode)
    c = bd.Pool(1, w.num_blocks, w.block_size, w.num_heads, w.head_dim, initial_free_order=w.free_order)
    o = ra.RefPool(w.num_blocks, [int(x) for x in w.free_order])
    B = w.block_size
    tc = np.full((w.num_seqs, w.max_blocks), -1, dtype=np.int32)
    lc = np.zeros(w.num_seqs, dtype=np.int32)
    to = [[-1] * w.max_blocks for _ in range(w.num_seqs)]
    lo = [0] * w.num_seqs
    dc, do = {}, {}
    for op in w.script:
        if op[0] == "admit":
            _, s, T = op
            nb = -(-T // B)
            tc[s, :nb] = c.alloc(nb)
            lc[s] = T
            to[s] = ra.admit(o, T, B, w.max_blocks)
            lo[s] = T
        elif op[0] == "fork":
            _, a, b = op
            nb = -(-int(lc[a]) // B)
            c.incref(tc[a, :nb])
            tc[b] = tc[a]
            lc[b] = lc[a]
            to[b] = ra.fork(o, to[a], lo[a], B)
            lo[b] = lo[a]
        elif op[0] == "dummy_alloc":
            dc[op[1]] = c.alloc(op[2])
            do[op[1]] = o.alloc(op[2])
        elif op[0] == "dummy_free":
            c.free(dc.pop(op[1]))
            o.free(do.pop(op[1]))
        elif op[0] == "write":
            sc, pc = c.prepare_append(tc, lc, op[1])
            so, po = o.prepare_append(to, lo, op[1], B, w.max_blocks)
            assert sc.tolist() == so and [tuple(p) for p in pc.tolist()] == po
        elif op[0] == "prompt":
            _, s, tokens = op
            hc_, ho_ = bd.prompt_block_hashes(tokens, B), ra.prompt_block_hashes(tokens, B)
            assert hc_ == ho_
            hit_c, hit_o = c.prefix_lookup(hc_), o.prefix_lookup(ho_)
            assert hit_c == hit_o
            tc[s, :len(hit_c)] = hit_c
            lc[s] = len(hit_c) * B
            to[s] = hit_o + [-1] * (w.max_blocks - len(hit_o))
            lo[s] = len(hit_o) * B
            counts = [0] * w.num_seqs
            counts[s] = len(tokens) - len(hit_o) * B
            sc, pc = c.prepare_append(tc, lc, counts)
            so, po = o.prepare_append(to, lo, counts, B, w.max_blocks)
            assert sc.tolist() == so
            c.prefix_register(hc_[len(hit_c):], tc[s, len(hit_c):len(hc_)])
            o.prefix_register(ho_[len(hit_o):], to[s][len(hit_o):len(ho_)])
        assert tc.tolist() == to and lc.tolist() == lo
    # a few decode steps
    for _ in range(3):
        sc, pc = c.prepare_append(tc, lc)
        so, po = o.prepare_append(to, lo, [1] * w.num_seqs, B, w.max_blocks)
        assert sc.tolist() == so and [tuple(p) for p in pc.tolist()] == po
        assert tc.tolist() == to and lc.tolist() == lo
    _same(c, o)
    if index == 4:
        st = c.stats()
        assert abs(st["used_blocks"] / w.num_blocks - 0.9) < 0.02


def test_prepare_append_failure_changes_nothing():
    c = bd.Pool(1, 3, 8, 1, 64)
    ids = c.alloc(1)
    c.incref(ids)
    tables = np.array([[ids[0], -1, -1], [ids[0], -1, -1]], dtype=np.int32)
    lens = np.array([4, 4], dtype=np.int32)
    q0 = c.free_queue()
    with pytest.raises(pkv.PkvError) as e:
        c.prepare_append(tables, lens, [9, 9])       # 2 COW + 2 new blocks > 2 free
    assert e.value.code == "OUT_OF_BLOCKS"
    assert tables.tolist() == [[ids[0], -1, -1], [ids[0], -1, -1]] and lens.tolist() == [4, 4]
    assert c.free_queue() == q0 and c.refcount(ids[0]) == 2 and c.stats()["cow_copies"] == 0
    c.validate()


def test_device_ops_refuse_host_only_pool():
    c = bd.Pool(1, 4, 8, 1, 64)
    rc = pkv.lib().pkv_append(c.handle, 0, None, None, None, 1, None, None)
    assert rc == 1 and "device memory" in pkv.last_error()
    rc = pkv.lib().pkv_copy_blocks(c.handle, None, 1, None, None)
    assert rc == 1


def test_launch_info_checks_arguments_before_any_cuda_call():
    for args in ((32, 96, 0), (-1, 128, 0), (5000, 128, 0), (32, 128, 2), (32, 128, -1)):
        rc = pkv.lib().pkv_decode_launch_info(*args, None, None, None)
        assert rc == 1, args
    with pytest.raises(pkv.PkvError) as e:
        pkv.decode_launch_info(32, 128, "bf16")
    assert e.value.code == "INVALID_ARG"


# ------------------------------------------------------------------ prefix cache: library vs oracle

def test_block_hash_matches_oracle():
    rng = random.Random(5)
    for _ in range(200):
        parent = rng.randrange(1 << 64)
        toks = [rng.randrange(-2**31, 2**31) for _ in range(rng.randrange(0, 40))]
        assert bd.block_hash(parent, toks) == ra.block_hash(parent, toks)
    toks = [rng.randrange(32000) for _ in range(100)]
    assert bd.prompt_block_hashes(toks, 16) == ra.prompt_block_hashes(toks, 16)


def test_prompt_block_hashes_matches_oracle():
    """pkv_prompt_block_hashes chains the per-block hashes in the library: equal to the oracle's
    chain for every block size, prompt lengths with and without a partial last block, and empty."""
    rng = random.Random(11)
    for B in (1, 8, 16, 32, 256):
        for n in (0, B - 1, B, 3 * B + 5, 40 * B):
            toks = [rng.randrange(-2**31, 2**31) for _ in range(n)]
            assert bd.prompt_block_hashes(toks, B) == ra.prompt_block_hashes(toks, B), (B, n)


def test_prompt_block_hashes_argument_errors():
    L = bd.lib()
    toks = np.arange(64, dtype=np.int32)
    out = np.zeros(4, dtype=np.uint64)
    n = ctypes.c_int32(-7)
    # capacity below the number of full blocks: refused, nothing written
    assert L.pkv_prompt_block_hashes(toks.ctypes.data, 64, 16, out.ctypes.data, 3, ctypes.byref(n)) == 1
    assert n.value == -7 and not out.any()
    assert L.pkv_prompt_block_hashes(toks.ctypes.data, 64, 0, out.ctypes.data, 4, ctypes.byref(n)) == 1
    assert L.pkv_prompt_block_hashes(toks.ctypes.data, -1, 16, out.ctypes.data, 4, ctypes.byref(n)) == 1
    assert L.pkv_prompt_block_hashes(toks.ctypes.data, 64, 16, out.ctypes.data, 4, None) == 1
    assert L.pkv_prompt_block_hashes(toks.ctypes.data, 64, 16, out.ctypes.data, 4, ctypes.byref(n)) == 0
    assert n.value == 4 and [int(x) for x in out] == ra.prompt_block_hashes(toks.tolist(), 16)


def _same_prefix_state(c, o):
    _same(c, o)
    st, so = c.stats(), o.stats()
    assert (st["cached_blocks"], st["cached_free_blocks"], st["prefix_hits"], st["prefix_misses"],
            st["evictions"]) == (so.cached_blocks, so.cached_free_blocks, so.prefix_hits, so.prefix_misses,
                                 so.evictions)


@pytest.mark.parametrize("seed", range(8))
def test_prefix_cache_matches_oracle(seed):
    rng = random.Random(100 + seed)
    B, N, maxb = 8, 20, 8
    order = rng.sample(range(N), N)
    c = bd.Pool(1, N, B, 1, 64, initial_free_order=order)
    o = ra.RefPool(N, order)
    prefixes = [[rng.randrange(40) for _ in range(24)] for _ in range(3)]
    live = {}
    for step in range(160):
        r = rng.random()
        if live and r < 0.3:
            k = rng.choice(sorted(live))
            ids = live.pop(k)
            _both(lambda: c.free(ids), lambda: o.free(ids))
        elif r < 0.4:
            ids = [rng.randrange(-1, N + 1) for _ in range(2)]
            hs = [rng.randrange(1 << 64) for _ in range(2)]
            _both(lambda: c.prefix_register(hs, ids), lambda: o.prefix_register(hs, ids))
        else:
            toks = rng.choice(prefixes)[: rng.randrange(8, 25)] + [rng.randrange(40) for _ in range(rng.randrange(9))]
            hs = ra.prompt_block_hashes(toks, B)
            hc, ho = _both(lambda: c.prefix_lookup(hs), lambda: o.prefix_lookup(hs))
            assert hc == ho
            need = -(-len(toks) // B) - len(ho)
            nc, no = _both(lambda: c.alloc(need), lambda: o.alloc(need))
            if no is None:
                _both(lambda: c.free(ho), lambda: o.free(ho))
            else:
                assert nc == no
                ids = ho + no
                _both(lambda: c.prefix_register(hs[len(ho):], ids[len(ho):len(hs)]),
                      lambda: o.prefix_register(hs[len(ho):], ids[len(ho):len(hs)]))
                live[step] = ids
        _same_prefix_state(c, o)
    # appends that take cached free blocks evict them in both, and roll back alike on failure
    tables_c = np.full((1, maxb), -1, dtype=np.int32)
    lens_c = np.zeros(1, dtype=np.int32)
    tables_o, lens_o = [[-1] * maxb], [0]
    for n in (3, 20, 200):
        rc, ro = _both(lambda: c.prepare_append(tables_c, lens_c, [n]),
                       lambda: o.prepare_append(tables_o, lens_o, [n], B, maxb))
        assert tables_c.tolist() == tables_o and lens_c.tolist() == lens_o
        _same_prefix_state(c, o)


def test_package_import_fails_loudly_without_the_library(tmp_path):
    """A copy of the package with no libpkv.so next to it refuses to import (there is no CPU or
    library fallback)."""
    import shutil
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "paged_kv_cache_88_gb300")
    dst = tmp_path / "paged_kv_cache_88_gb300"
    shutil.copytree(pkg, dst, ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc"))
    shutil.copytree(os.path.join(root, "workloads"), tmp_path / "workloads")
    r = subprocess.run([sys.executable, "-c", "import paged_kv_cache_88_gb300"], capture_output=True, text=True,
                       cwd=str(tmp_path), timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libpkv.so" in r.stderr
