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


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle timed on the host cores) prints one JSON line
    with the contract's keys, on the GPU arm's workload, metric and unit, no host-device
    bytes, and its own run described in cpu_baseline."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["config"]["workload"] == "cfg2-7b"
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
