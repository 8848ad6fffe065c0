"""Host-side pieces of bench.py that need no GPU: the oracle's timed CPU baseline
(all cores and one core) and the CPU model string it reports."""
import numpy as np

import bench
import workloads as wl


def _layer(w, seed=0):
    rng = np.random.default_rng(seed)
    N, B, H, D = w.num_blocks, w.block_size, w.num_heads, w.head_dim
    shape = (N, H, B, D) if w.layout == "HND" else (N, B, H, D)
    k = rng.standard_normal(shape).astype(np.float16)
    v = rng.standard_normal(shape).astype(np.float16)
    lens = np.asarray(w.context_lens, dtype=np.int32)
    tables = np.zeros((w.num_seqs, w.max_blocks), dtype=np.int32)
    perm, i = rng.permutation(N), 0
    for s, t in enumerate(lens):
        nb = -(-int(t) // B)
        tables[s, :nb] = perm[i:i + nb]
        i += nb
    return k, v, tables, lens


def test_cpu_baseline_reports_all_cores_and_one_core():
    w = wl.make_workload(2, num_layers=1, num_seqs=8, len_scale=0.05, decode_steps=1)
    k, v, tables, lens = _layer(w)
    r = bench.cpu_baseline_oracle(w, k, v, tables, lens, 0.2)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s"
    assert r["cores"] >= 1 and r["value"] > 0 and r["one_core_value"] > 0
    assert isinstance(r["cpu_model"], str) and r["cpu_model"]
    assert "one core" in r["sample"]
    # the one-core sample must not leave the oracle pinned to one thread
    from oracle import ref_attn_c as rc
    assert rc.max_threads() == r["cores"]


def test_cpu_model_is_a_name():
    m = bench.cpu_model()
    assert isinstance(m, str) and len(m) > 0
