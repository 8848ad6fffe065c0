"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by element.

Bar: block tables, slots, COW pairs and every pool byte after append / copy are
bit-exact; attention outputs satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref| against the
float64 oracle (fp16 K/V with fp32 accumulation, fp16 output).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_88_gb300 as pkv  # noqa: E402
from paged_kv_cache_88_gb300.engine import DecodeEngine  # noqa: E402
from oracle import ref_attn as rf  # noqa: E402
from oracle import ref_attn_c as rc  # noqa: E402
from oracle.driver import OracleEngine  # noqa: E402
import workloads as wl  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    gpu = gpu.astype(np.float64)
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu {gpu[i]} ref {ref[i]} err {err[i]:.3e}")


def u16(t):
    return t.detach().cpu().numpy().view(np.uint16)


def bits(t):
    a = t.detach().cpu().numpy()
    return a.view(np.uint8 if a.dtype == np.uint8 else (np.uint16 if a.itemsize == 2 else np.uint32))


def same_pools(eng, ora, what=""):
    """Every pool byte (and, for an E4M3 cache, every scale) equal to the oracle's."""
    assert np.array_equal(bits(eng.k_pool), ora.k_pool.view(bits(eng.k_pool).dtype)), f"K pool differs {what}"
    assert np.array_equal(bits(eng.v_pool), ora.v_pool.view(bits(eng.v_pool).dtype)), f"V pool differs {what}"
    if eng.k_scale is not None:
        assert np.array_equal(bits(eng.k_scale), ora.k_scale.view(np.uint32)), f"K scales differ {what}"
        assert np.array_equal(bits(eng.v_scale), ora.v_scale.view(np.uint32)), f"V scales differ {what}"


def make_oracle(w):
    if w.kv_dtype == "e4m3":
        return OracleEngine(w, wl.pool_codes_e4m3(w, 0), wl.pool_codes_e4m3(w, 1), wl.pool_scales(w, 0),
                            wl.pool_scales(w, 1))
    return OracleEngine(w, wl.pool_values(w, 0), wl.pool_values(w, 1))


def run_parity(w, steps: int, fused: bool = True, cascade: bool = True):
    eng = DecodeEngine(w, fill="numpy", fused=fused, cascade=cascade)
    ora = make_oracle(w)
    eng.run_script(values="numpy")
    ora.run_script()
    torch.cuda.synchronize()
    assert eng.tables.tolist() == ora.tables and eng.lens.tolist() == ora.lens
    same_pools(eng, ora, "after set-up")
    for step in range(steps):
        q, k, v = ora.step_inputs(step)
        qd, kd, vd = eng.step_inputs(step, "numpy")
        out = torch.empty_like(qd)
        eng.step(qd, kd, vd, out)
        torch.cuda.synchronize()
        ref = ora.step(q, k, v)
        assert eng.device_status() == 0
        assert eng.last_slots.tolist() == ora.last_slots
        assert [tuple(p) for p in eng.last_pairs.tolist()] == ora.last_pairs
        assert eng.tables.tolist() == ora.tables and eng.lens.tolist() == ora.lens
        same_pools(eng, ora, f"after step {step}")
        assert_close(out.cpu().numpy(), ref, f"{w.name} step {step}")
        assert eng.device_status() == 0
    eng.pool.validate()
    return eng, ora


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_tiny_config(layout):
    w = wl.make_workload(1, layout=layout, decode_steps=3)
    eng, _ = run_parity(w, 3)
    # 64 -> 65 -> 66 -> 67 tokens: the block boundary at 64 took a fresh block
    assert eng.lens.tolist() == [20, 36, 53, 67]


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("fused", [True, False])
def test_7b_shape_reduced(layout, fused):
    """The decode step with the append fused into the attention launch, and with two launches."""
    w = wl.make_workload(2, num_layers=2, num_seqs=8, len_scale=0.3, decode_steps=3, layout=layout)
    run_parity(w, 3, fused=fused)


@pytest.mark.parametrize("cascade", [True, False])
@pytest.mark.parametrize("fused", [True, False])
def test_prefix_sharing_cow_reduced(cascade, fused):
    """The forked prompt: with the cascade (prefix pass + private pass) and without."""
    w = wl.make_workload(3, num_layers=2, num_seqs=8, len_scale=0.25, decode_steps=3)
    eng, ora = run_parity(w, 3, fused=fused, cascade=cascade)
    assert (eng.plan_groups == 1) == cascade
    st = eng.pool.stats()
    assert st["cow_copies"] == w.num_seqs - 1


def test_prefix_found_by_block_hash_reduced():
    """Requests arriving with the same prompt tokens share its full blocks through the prefix cache."""
    w = wl.make_workload(3, num_layers=2, num_seqs=8, len_scale=0.25, decode_steps=3, prefix_mode="hash")
    eng, ora = run_parity(w, 3)
    st = eng.pool.stats()
    shared_full = 130 // w.block_size                  # 0.25 x 520 prompt tokens -> 8 full blocks
    assert st["prefix_hits"] == (w.num_seqs - 1) * shared_full
    assert st["cow_copies"] == 0
    so = ora.pool.stats()
    assert (st["prefix_hits"], st["prefix_misses"], st["cached_blocks"]) == \
        (so.prefix_hits, so.prefix_misses, so.cached_blocks)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_13b_shape_churned_pool_reduced(layout):
    w = wl.make_workload(4, num_layers=2, num_seqs=24, len_scale=0.5, decode_steps=2, layout=layout)
    run_parity(w, 2)


@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128, 256, 512])
def test_long_context_block_sweep_reduced(block_size):
    w = wl.make_workload(5, num_layers=1, num_seqs=3, len_scale=0.12, decode_steps=2, block_size=block_size)
    run_parity(w, 2)


# ----------------------------------------------------------------------------- swap (preemption)

@pytest.mark.parametrize("kv_dtype,direct", [("f16", False), ("e4m3", False), ("f16", True), ("e4m3", True)])
def test_swap_out_and_in_round_trip(kv_dtype, direct):
    """Two sequences are swapped to pinned host memory, their blocks reused by other requests,
    then swapped back into new blocks; the next decode step matches the oracle exactly.
    direct: the kernels read and write the pinned host buffers themselves (no device staging)."""
    w = wl.make_workload(2, num_layers=2, num_seqs=6, len_scale=0.2, decode_steps=4, kv_dtype=kv_dtype)
    eng = DecodeEngine(w, fill="numpy")
    ora = make_oracle(w)
    eng.run_script()
    ora.run_script()
    q, k, v = ora.step_inputs(0)
    qd, kd, vd = eng.step_inputs(0)
    out = torch.empty_like(qd)
    eng.step(qd, kd, vd, out)
    ora.step(q, k, v)
    bpb = eng.pool.swap_bytes_per_block()
    host = torch.empty(64 * bpb, dtype=torch.uint8).pin_memory()
    staging = None if direct else torch.empty(64 * bpb, dtype=torch.uint8, device="cuda")
    host2 = torch.empty_like(host).pin_memory()
    n1 = eng.swap_out(1, host, staging)
    torch.cuda.synchronize()
    n3 = eng.swap_out(3, host2, staging)
    s1, s3 = ora.swap_out(1), ora.swap_out(3)
    # other requests take every free block (the freed ones included), scribble on them and finish
    nfree = eng.pool.stats()["free_blocks"]
    junk = eng.pool.alloc(nfree)
    ora_junk = ora.pool.alloc(nfree)
    assert junk == ora_junk
    torch.cuda.synchronize()
    jb = torch.tensor(junk, dtype=torch.int32, device="cuda")
    scribble = torch.full((len(junk) * bpb,), 0x55, dtype=torch.uint8, device="cuda")
    eng.pool.scatter_blocks(jb, scribble)
    for a in ora._arrays():
        a[:, ora_junk] = np.frombuffer(b"\x55" * a[:, ora_junk].nbytes, dtype=a.dtype).reshape(a[:, ora_junk].shape)
    eng.pool.free(junk)
    ora.pool.free(ora_junk)
    eng.swap_in(1, n1, host, staging)
    torch.cuda.synchronize()
    eng.swap_in(3, n3, host2, staging)
    ora.swap_in(1, s1)
    ora.swap_in(3, s3)
    torch.cuda.synchronize()
    assert eng.tables.tolist() == ora.tables
    same_pools(eng, ora, "after swap")
    eng.upload_tables()
    q, k, v = ora.step_inputs(1)
    qd, kd, vd = eng.step_inputs(1)
    eng.step(qd, kd, vd, out)
    torch.cuda.synchronize()
    ref = ora.step(q, k, v)
    assert eng.device_status() == 0
    same_pools(eng, ora, "after the step")
    assert_close(out.cpu().numpy(), ref, "after swap")


def test_swap_refuses_pageable_host_buffer():
    """A buffer the device cannot address (pageable host memory) is refused before any launch."""
    w = wl.make_workload(2, num_layers=2, num_seqs=2, len_scale=0.1, decode_steps=1)
    eng = DecodeEngine(w, fill="numpy")
    eng.run_script()
    bpb = eng.pool.swap_bytes_per_block()
    blocks = torch.tensor(eng.tables[0, :1], dtype=torch.int32, device="cuda")
    pageable = torch.empty(bpb, dtype=torch.uint8)
    with pytest.raises(pkv.PkvError) as ei:
        eng.pool.gather_blocks(blocks, pageable)
    assert ei.value.code == "INVALID_ARG"
    with pytest.raises(pkv.PkvError):
        eng.pool.scatter_blocks(blocks, pageable)
    torch.cuda.synchronize()
    assert eng.device_status() == 0


# ----------------------------------------------------------------------------- FP8 E4M3 cache

@pytest.mark.parametrize("fused", [True, False])
def test_e4m3_tiny(fused):
    """head_dim 64; codes and scales written by the quantising append are bit-exact."""
    w = wl.make_workload(1, decode_steps=3, kv_dtype="e4m3")
    run_parity(w, 3, fused=fused)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("fused", [True, False])
def test_e4m3_7b_shape_reduced(fused, layout):
    w = wl.make_workload(2, num_layers=2, num_seqs=8, len_scale=0.3, decode_steps=3, kv_dtype="e4m3", layout=layout)
    run_parity(w, 3, fused=fused)


@pytest.mark.parametrize("fused", [True, False])
def test_e4m3_nhd_tiny_and_long(fused):
    """The E4M3 cache in the NHD layout: head_dim 64 (tiny workload) and long contexts at
    block sizes 8 and 256; codes and scales bit-exact, attention against the oracle."""
    run_parity(wl.make_workload(1, decode_steps=3, kv_dtype="e4m3", layout="NHD"), 3, fused=fused)
    for bs in (8, 256):
        w = wl.make_workload(5, num_layers=1, num_seqs=3, len_scale=0.12, decode_steps=2, block_size=bs,
                             kv_dtype="e4m3", layout="NHD")
        run_parity(w, 2, fused=fused)


def test_e4m3_prefix_cow_reduced():
    """COW copies the codes and the row scales of the shared block."""
    w = wl.make_workload(3, num_layers=2, num_seqs=8, len_scale=0.25, decode_steps=2, kv_dtype="e4m3")
    eng, _ = run_parity(w, 2)
    assert eng.pool.stats()["cow_copies"] == w.num_seqs - 1


def test_e4m3_13b_shape_reduced():
    w = wl.make_workload(4, num_layers=2, num_seqs=24, len_scale=0.5, decode_steps=2, kv_dtype="e4m3")
    run_parity(w, 2)


@pytest.mark.parametrize("block_size", [8, 16, 32, 64, 128, 256, 512])
def test_e4m3_long_context_reduced(block_size):
    w = wl.make_workload(5, num_layers=1, num_seqs=3, len_scale=0.12, decode_steps=2, block_size=block_size,
                         kv_dtype="e4m3")
    run_parity(w, 2)


def test_e4m3_pool_rules():
    q = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.Pool(1, 1, 16, 1, 256, "HND", kv_dtype="e4m3")          # head_dim 256 not built for E4M3
    assert e.value.code == "UNSUPPORTED"
    pkv.Pool(1, 1, 16, 1, 64, "NHD", kv_dtype="e4m3")                # either layout
    p = pkv.Pool(1, 1, 8, 1, 64, "HND", k_pool=torch.zeros(512, dtype=torch.uint8, device="cuda"),
                 v_pool=torch.zeros(512, dtype=torch.uint8, device="cuda"), kv_dtype="e4m3")
    kn = torch.zeros((1, 1, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:                          # no scale pools attached
        p.append(0, kn, kn, torch.zeros(1, dtype=torch.int64, device="cuda"))
    assert "scale" in pkv.last_error()
    del q


def test_e4m3_row_scales_over_many_octaves():
    """V row scales from 2^-40 to 2^6 within one sequence, a sequence whose V scales are
    all tiny, a zero row (codes 0, scale 1), a row whose V scale is 0, one-token and empty
    contexts, and NaN codes and scales past every context (never read): the attention of
    code x scale, each (sequence, head) within the usual 2e-3 abs + 1e-2 rel taken
    relative to its largest output (plus the fp16 subnormal step)."""
    from oracle import fp8
    rng = np.random.default_rng(41)
    H, D, B = 2, 128, 16
    lens = [37, 200, 513, 1, 0]
    nb = [-(-t // B) for t in lens]
    N = sum(nb) + 3
    perm = rng.permutation(N)
    tab = np.zeros((len(lens), max(nb)), dtype=np.int32)
    i = 0
    for s_, n_ in enumerate(nb):
        tab[s_, :n_] = perm[i:i + n_]
        i += n_
    kc = rng.integers(0, 256, size=(N, H, B, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(N, H, B, D), dtype=np.uint8)
    for c_ in (kc, vc):
        c_[(c_ & 0x7F) == 0x7F] ^= 1                       # no NaN codes inside the contexts
    ks = np.exp2(rng.uniform(-7, -5, size=(N, H, B))).astype(np.float32)
    vs = np.exp2(rng.uniform(-40, 6, size=(N, H, B))).astype(np.float32)
    lo = {1: (-22, -20), 2: (-2, 6), 3: (-30, -30)}
    for s_, T in enumerate(lens):
        for t in range(T):
            b_, o_ = tab[s_, t // B], t % B
            if s_ in lo:
                vs[b_, :, o_] = np.exp2(rng.uniform(*lo[s_], size=H))
        if T % B:                                          # past the context: NaN codes and scales
            b_ = tab[s_, T // B]
            kc[b_, :, T % B:] = 0x7F
            vc[b_, :, T % B:] = 0xFF
            ks[b_, :, T % B:] = np.nan
            vs[b_, :, T % B:] = np.nan
    b_, o_ = tab[2, 100 // B], 100 % B                     # a zero row
    kc[b_, :, o_] = 0
    vc[b_, :, o_] = 0
    ks[b_, :, o_] = 1.0
    vs[b_, :, o_] = 1.0
    b_, o_ = tab[2, 300 // B], 300 % B                     # a V scale of 0
    vs[b_, :, o_] = 0.0
    q = rng.standard_normal((len(lens), H, D)).astype(np.float16)
    dev = "cuda"
    pool = pkv.Pool(1, N, B, H, D, "HND", k_pool=torch.from_numpy(kc).to(dev), v_pool=torch.from_numpy(vc).to(dev),
                    kv_dtype="e4m3", k_scale=torch.from_numpy(ks).to(dev), v_scale=torch.from_numpy(vs).to(dev))
    qd = torch.from_numpy(q).to(dev)
    out = torch.full_like(qd, float("nan"))
    ws = pkv.new_workspace(len(lens), H, D, dev)
    pool.decode_attention(0, qd, torch.from_numpy(tab).to(dev), torch.from_numpy(np.array(lens, dtype=np.int32)).to(dev),
                          out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    ref = fp8.decode_attention(q, kc, vc, ks, vs, tab, np.array(lens), B)
    assert np.all(got[4] == 0)
    for s_ in range(len(lens) - 1):
        for h in range(H):
            big = np.abs(ref[s_, h]).max()
            err = np.abs(got[s_, h] - ref[s_, h])
            assert (err <= 2e-3 * big + 1e-2 * np.abs(ref[s_, h]) + 6e-8).all(), \
                (s_, h, float(err.max()), float(big))


# ----------------------------------------------------------------------------- raw-call edge cases

def _raw_case(lens, H=3, D=128, B=16, N=None, seed=0, layout="NHD", canary_nan=True):
    rng = np.random.default_rng(seed)
    S = len(lens)
    nb = [-(-t // B) for t in lens]
    N = N or sum(nb) + 5
    perm = rng.permutation(N)
    maxb = max(nb + [1])
    tables = np.zeros((S, maxb), dtype=np.int32)
    i = 0
    for s in range(S):
        for j in range(nb[s]):
            tables[s, j] = perm[i]
            i += 1
    shape = (N, B, H, D) if layout == "NHD" else (N, H, B, D)
    if canary_nan:
        kp = np.full(shape, np.uint16(0x7E00), dtype=np.uint16).view(np.float16)   # NaN everywhere ...
        vp = kp.copy()
        for s, t in enumerate(lens):                                               # ... but valid tokens
            for tok in range(t):
                blk, off = tables[s, tok // B], tok % B
                idx = (blk, off) if layout == "NHD" else (blk, slice(None), off)
                kp[idx] = rng.standard_normal((H, D)).astype(np.float16)
                vp[idx] = rng.standard_normal((H, D)).astype(np.float16)
    else:
        kp = rng.standard_normal(shape).astype(np.float16)
        vp = rng.standard_normal(shape).astype(np.float16)
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    return q, kp, vp, tables, np.asarray(lens, dtype=np.int32), B, N


def _gpu_attn(q, kp, vp, tables, lens, B, N, layout="NHD", scale=0.0, ws=None):
    dev = "cuda"
    qd = torch.from_numpy(q).to(dev)
    kd = torch.from_numpy(kp).to(dev)
    vd = torch.from_numpy(vp).to(dev)
    td = torch.from_numpy(tables).to(dev)
    ld = torch.from_numpy(lens).to(dev)
    if ws is None:
        ws = pkv.new_workspace(q.shape[0], q.shape[1], q.shape[2], dev)
    out = pkv.decode_attention(qd, kd, vd, td, ld, num_blocks=N, block_size=B, layout=layout, scale=scale,
                               workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), pkv.workspace_status(ws), ws


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_edge_lengths_with_nan_canary(layout):
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 64, 100, 257]
    q, kp, vp, tab, ln, B, N = _raw_case(lens, layout=layout)
    out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N, layout)
    assert st == 0
    assert np.isfinite(out).all()
    assert np.all(out[0] == 0)          # empty context
    ref = rf.decode_attention(q, kp, vp, tab, ln, B, layout)
    assert_close(out, ref, "edge lengths")
    # T = 1: out is V[0] rounded to fp16
    blk = tab[1, 0]
    v0 = vp[blk, 0] if layout == "NHD" else vp[blk, :, 0]
    assert np.array_equal(out[1].astype(np.float16).view(np.uint16), v0.view(np.uint16))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_head_dims(D):
    q, kp, vp, tab, ln, B, N = _raw_case([5, 77, 300, 129], H=2, D=D, canary_nan=False, seed=D)
    out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N)
    assert st == 0
    assert_close(out, rc.decode_attention(q, kp, vp, tab, ln, B), f"D={D}")


def test_explicit_scale():
    q, kp, vp, tab, ln, B, N = _raw_case([40, 90], H=2, canary_nan=False, seed=3)
    out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N, scale=0.05)
    assert st == 0
    assert_close(out, rf.decode_attention(q, kp, vp, tab, ln, B, scale=0.05), "scale 0.05")


def test_one_long_sequence_spans_every_cta():
    """One (s, h) split over all CTAs of the launch: the fused combine merges hundreds of pieces."""
    q, kp, vp, tab, ln, B, N = _raw_case([40000], H=1, B=256, canary_nan=False, seed=5)
    out, st, ws = _gpu_attn(q, kp, vp, tab, ln, B, N)
    assert st == 0
    assert_close(out, rc.decode_attention(q, kp, vp, tab, ln, B), "long")
    out2, st2, _ = _gpu_attn(q, kp, vp, tab, ln, B, N, ws=ws)   # counters were reset: same result
    assert st2 == 0 and np.array_equal(out, out2)


@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_very_long_sequence_small_blocks(layout):
    """One 65,536-token sequence in 8-token blocks beside a short one: an 8,192-entry block
    table (the producer's 128-entry window refilled 64 times per (sequence, head)), blocks
    scattered over the pool, every CTA of the launch on the long sequence's pieces."""
    q, kp, vp, tab, ln, B, N = _raw_case([65536, 100], H=2, B=8, canary_nan=True, seed=9, layout=layout)
    out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N, layout)
    assert st == 0
    assert_close(out, rc.decode_attention(q, kp, vp, tab, ln, B, layout), f"65536 tokens B=8 {layout}")


def test_workspace_reused_across_batch_sizes():
    """One workspace, sized for 48 sequences of 8 heads, serves calls with 6, then 48, then 20
    sequences and then another head_dim. The small batch's (s, h) are split over many CTAs,
    so its pieces fill the workspace; the counters of the larger batches must still start
    at zero, so their place may not depend on num_seqs."""
    H = 8
    ws = pkv.new_workspace(48, H, 128, "cuda")
    for S, D, seed in ((6, 128, 21), (48, 128, 22), (20, 128, 23), (48, 64, 24)):
        rng = np.random.default_rng(seed)
        lens = rng.integers(300, 2000, size=S).tolist()
        q, kp, vp, tab, ln, B, N = _raw_case(lens, H=H, D=D, canary_nan=False, seed=seed, layout="HND")
        out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N, layout="HND", ws=ws)
        assert st == 0
        assert_close(out, rc.decode_attention(q, kp, vp, tab, ln, B, "HND"), f"S={S} D={D}")


def test_many_short_sequences():
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 70, size=700).tolist()
    q, kp, vp, tab, ln, B, N = _raw_case(lens, H=4, D=64, B=8, canary_nan=False, seed=6)
    out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N)
    assert st == 0
    assert_close(out, rc.decode_attention(q, kp, vp, tab, ln, B), "many short")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_maximum_batch(layout):
    """The largest batch one launch takes (4096 sequences: the per-sequence lengths, starts
    and tile offsets fill the most shared memory), lengths 0..48 with empty contexts among
    them; one more sequence is refused."""
    rng = np.random.default_rng(31)
    lens = rng.integers(0, 49, size=4096).tolist()
    q, kp, vp, tab, ln, B, N = _raw_case(lens, H=2, D=128, B=16, canary_nan=False, seed=32, layout=layout)
    out, st, ws = _gpu_attn(q, kp, vp, tab, ln, B, N, layout)
    assert st == 0
    assert np.all(out[ln == 0] == 0)
    assert_close(out, rc.decode_attention(q, kp, vp, tab, ln, B, layout), f"4096 sequences {layout}")
    q1 = np.zeros((4097, 2, 128), dtype=np.float16)
    t1 = np.zeros((4097, tab.shape[1]), dtype=np.int32)
    with pytest.raises(pkv.binding.PkvError) as e:
        _gpu_attn(q1, kp, vp, t1, np.zeros(4097, dtype=np.int32), B, N, layout, ws=ws)
    assert e.value.code == "INVALID_ARG"


def test_bad_block_id_is_flagged_not_faulted():
    q, kp, vp, tab, ln, B, N = _raw_case([40, 20], H=2, canary_nan=False, seed=7)
    tab[0, 1] = N + 5            # out of range: the kernel clamps it and flags it
    out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N)
    assert st & pkv.DEV_BAD_BLOCK
    tab[0, 1] = -3
    _, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N)
    assert st & pkv.DEV_BAD_BLOCK
    # the context is fine afterwards
    q, kp, vp, tab, ln, B, N = _raw_case([40, 20], H=2, canary_nan=False, seed=7)
    out, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N)
    assert st == 0
    assert_close(out, rf.decode_attention(q, kp, vp, tab, ln, B), "after bad block")


def test_bad_length_is_flagged():
    q, kp, vp, tab, ln, B, N = _raw_case([40, 20], H=2, canary_nan=False, seed=8)
    ln[1] = tab.shape[1] * B + 7
    _, st, _ = _gpu_attn(q, kp, vp, tab, ln, B, N)
    assert st & pkv.DEV_BAD_LENGTH


def test_bad_slot_and_pair_are_flagged():
    w = wl.make_workload(1)
    eng = DecodeEngine(w, fill="numpy")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    k0 = eng.k_pool.clone()
    kn = torch.zeros((2, w.num_heads, w.head_dim), dtype=torch.float16, device="cuda")
    slots = torch.tensor([-1, w.num_blocks * w.block_size], dtype=torch.int64, device="cuda")
    eng.pool.append(0, kn, kn, slots, status=status)
    pairs = torch.tensor([[0, w.num_blocks]], dtype=torch.int32, device="cuda")
    eng.pool.copy_blocks(pairs, status=status)
    torch.cuda.synchronize()
    st = int(status[0].item())
    assert st & pkv.DEV_BAD_SLOT and st & pkv.DEV_BAD_PAIR
    assert torch.equal(eng.k_pool, k0)          # nothing was written


def test_fused_append_skip_and_bad_slot():
    """Slot -1: nothing stored, the pool row is used as it is; slot >= N*B: flagged, not stored."""
    w = wl.make_workload(1, decode_steps=2)
    eng = DecodeEngine(w, fill="numpy")
    ora = OracleEngine(w, wl.pool_values(w, 0), wl.pool_values(w, 1))
    eng.run_script()
    ora.run_script()
    q, k, v = ora.step_inputs(0)
    qd, kd, vd = eng.step_inputs(0)
    n_slots, n_pairs = eng.prepare_step()
    slots = eng.slots_d.clone()
    eng.slots_d[1] = -1
    eng.slots_d[2] = w.num_blocks * w.block_size + 3
    out = torch.empty_like(qd)
    eng.device_step(qd, kd, vd, out, n_slots, n_pairs)
    torch.cuda.synchronize()
    assert pkv.workspace_status(eng.workspace) & pkv.DEV_BAD_SLOT
    eng.workspace.zero_()
    # oracle: the same step with sequences 1 and 2 not written
    slots_o, pairs_o = ora.pool.prepare_append(ora.tables, ora.lens, [1] * w.num_seqs, w.block_size, w.max_blocks)
    assert slots_o == slots.tolist()
    slots_o[1] = -1
    slots_o[2] = -1
    rf.append_kv(ora.k_pool[0], ora.v_pool[0], k[0], v[0], slots_o, w.block_size, w.layout)
    ref = rf.decode_attention(q[0], ora.k_pool[0], ora.v_pool[0], ora.tables_array(), ora.lens, w.block_size,
                              w.layout)
    assert np.array_equal(u16(eng.k_pool), ora.k_pool.view(np.uint16))
    assert_close(out[0].cpu().numpy(), ref, "fused skip / bad slot")


@pytest.mark.parametrize("shape", ["tiny", "7b"])
def test_fused_append_skip_and_bad_slot_e4m3(shape):
    """E4M3 cache, append inside the attention launch: slot -1 stores nothing and the pool
    row (codes and scale) is read as it is; slot >= N*B is flagged and not stored (head_dim
    64 on the CUDA-core consumers, head_dim 128 on the tensor-core ones)."""
    from oracle import fp8
    if shape == "tiny":
        w = wl.make_workload(1, decode_steps=2, kv_dtype="e4m3")
    else:
        w = wl.make_workload(2, num_layers=1, num_seqs=6, len_scale=0.2, decode_steps=2, kv_dtype="e4m3")
    eng = DecodeEngine(w, fill="numpy", fused=True)
    ora = make_oracle(w)
    eng.run_script(values="numpy")
    ora.run_script()
    q, k, v = ora.step_inputs(0)
    qd, kd, vd = eng.step_inputs(0, "numpy")
    n_slots, n_pairs = eng.prepare_step()
    slots = eng.slots_d.clone()
    eng.slots_d[1] = -1
    eng.slots_d[2] = w.num_blocks * w.block_size + 3
    out = torch.empty_like(qd)
    eng.device_step(qd, kd, vd, out, n_slots, n_pairs)
    torch.cuda.synchronize()
    assert pkv.workspace_status(eng.workspace) & pkv.DEV_BAD_SLOT
    eng.workspace.zero_()
    slots_o, pairs_o = ora.pool.prepare_append(ora.tables, ora.lens, [1] * w.num_seqs, w.block_size, w.max_blocks)
    assert slots_o == slots.tolist()
    ora._copy(pairs_o)
    slots_o[1] = -1
    slots_o[2] = -1
    fp8.append_kv(ora.k_pool[0], ora.v_pool[0], ora.k_scale[0], ora.v_scale[0], k[0], v[0], slots_o,
                  w.block_size, w.layout)
    ref = fp8.decode_attention(q[0], ora.k_pool[0], ora.v_pool[0], ora.k_scale[0], ora.v_scale[0],
                               ora.tables_array(), ora.lens, w.block_size, layout=w.layout)
    assert np.array_equal(bits(eng.k_pool)[0], ora.k_pool[0].view(np.uint8))
    assert np.array_equal(bits(eng.v_pool)[0], ora.v_pool[0].view(np.uint8))
    assert np.array_equal(bits(eng.k_scale)[0], ora.k_scale[0].view(np.uint32))
    assert np.array_equal(bits(eng.v_scale)[0], ora.v_scale[0].view(np.uint32))
    assert_close(out[0].cpu().numpy(), ref, f"E4M3 fused skip / bad slot ({shape})")


def test_empty_batches_are_no_ops():
    """Zero sequences, tokens, pairs or chunks: each device entry point returns without a
    launch and leaves the pools and the status words as they were."""
    dev = "cuda"
    H, D, B, N = 2, 128, 16, 4
    kp = torch.randn((1, N, H, B, D), device=dev).half()
    vp = torch.randn((1, N, H, B, D), device=dev).half()
    k0, v0 = kp.clone(), vp.clone()
    pool = pkv.Pool(1, N, B, H, D, "HND", k_pool=kp, v_pool=vp)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = pkv.new_workspace(1, H, D)
    q = torch.zeros((0, H, D), dtype=torch.float16, device=dev)
    out = torch.zeros_like(q)
    tab = torch.zeros((0, 1), dtype=torch.int32, device=dev)
    lens = torch.zeros(0, dtype=torch.int32, device=dev)
    slots = torch.zeros(0, dtype=torch.int64, device=dev)
    pool.decode_attention(0, q, tab, lens, out, ws)
    pool.decode_append_attention(0, q, q, q, slots, tab, lens, out, ws)
    pool.append(0, q, q, slots, status=status)
    pool.copy_blocks(torch.zeros((0, 2), dtype=torch.int32, device=dev), status=status)
    pool.prefill_attention(0, q, torch.zeros(1, dtype=torch.int32, device=dev), 0, tab, lens, out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and pkv.workspace_status(ws) == 0
    assert torch.equal(kp, k0) and torch.equal(vp, v0)


def test_host_argument_errors():
    dev = "cuda"
    q = torch.zeros((2, 2, 96), dtype=torch.float16, device=dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.decode_attention(q, q, q, torch.zeros((2, 1), dtype=torch.int32, device=dev),
                             torch.zeros(2, dtype=torch.int32, device=dev), num_blocks=1, block_size=16,
                             workspace=torch.zeros(1 << 20, dtype=torch.uint8, device=dev))
    assert e.value.code in ("UNSUPPORTED", "INVALID_ARG")
    q = torch.zeros((2, 2, 128), dtype=torch.float16, device=dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.decode_attention(q, q, q, torch.zeros((2, 1), dtype=torch.int32, device=dev),
                             torch.zeros(2, dtype=torch.int32, device=dev), num_blocks=1, block_size=16,
                             workspace=torch.zeros(64, dtype=torch.uint8, device=dev))
    assert e.value.code == "INVALID_ARG" and "workspace" in pkv.last_error()


# ----------------------------------------------------------------------------- full size

@pytest.fixture
def free_gpu_memory():
    yield
    import gc
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_7b_full_size_bench_launch_sampled(layout, free_gpu_memory):
    """The 7B-shape batch-32 workload at full size, 32 layers, in the benchmark's launch configuration
    (the default HND pools, and NHD as `bench.py --layout NHD` runs it).

    The oracle allocator replays the same script (tables bit-exact); for two
    layers the pre-step pools are read back and the float64 C oracle computes
    every (sequence, head) of the step.
    """
    w = wl.make_workload(2, layout=layout)
    eng = DecodeEngine(w, fill="torch")
    eng.run_script()
    from oracle import ref_alloc as ra
    op = ra.RefPool(w.num_blocks, [int(x) for x in w.free_order])
    tabs = [ra.admit(op, int(t), w.block_size, w.max_blocks) for t in w.context_lens]
    lens = [int(t) for t in w.context_lens]
    assert eng.tables.tolist() == tabs
    qd, kd, vd = eng.step_inputs(0, "torch")
    check_layers = [0, w.num_layers - 1]
    before = {l: (eng.k_pool[l].cpu().numpy(), eng.v_pool[l].cpu().numpy()) for l in check_layers}
    out = torch.empty_like(qd)
    eng.step(qd, kd, vd, out)
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    slots, pairs = op.prepare_append(tabs, lens, [1] * w.num_seqs, w.block_size, w.max_blocks)
    assert eng.last_slots.tolist() == slots and pairs == []
    assert eng.tables.tolist() == tabs
    tab = np.asarray(tabs, dtype=np.int32)
    for l in check_layers:
        kp, vp = before[l]
        rf.append_kv(kp, vp, kd[l].cpu().numpy(), vd[l].cpu().numpy(), slots, w.block_size, w.layout)
        assert np.array_equal(kp.view(np.uint16), u16(eng.k_pool[l]))
        ref = rc.decode_attention(qd[l].cpu().numpy(), kp, vp, tab, np.asarray(lens, dtype=np.int32),
                                  w.block_size, w.layout)
        assert_close(out[l].cpu().numpy(), ref, f"7b full layer {l}")


def _full_size(w, check_layers, steps: int = 2):
    """Full-size workload through the engine (torch-made pools); oracle on the listed layers.

    The oracle replays the same host script with its own allocator (tables,
    slots and COW pairs bit-exact), starts from the pools read back before any
    write, applies its own copies and appends, and computes every (sequence,
    head) of each step with the float64 C oracle.
    """
    import dataclasses
    eng = DecodeEngine(w, fill="torch")
    snap_k = np.stack([eng.k_pool[l].cpu().numpy() for l in check_layers])
    snap_v = np.stack([eng.v_pool[l].cpu().numpy() for l in check_layers])
    eng.run_script(values="torch")
    sub = dataclasses.replace(w, num_layers=len(check_layers))
    ora = OracleEngine(sub, snap_k, snap_v)
    del snap_k, snap_v

    def values(op_index, i, which, n):
        layer = check_layers[i]
        return wl.torch_normal_fp16(w.seed, (400 + which, op_index, layer), (n, w.num_heads, w.head_dim),
                                    "cuda").cpu().numpy()

    ora.run_script(values)
    torch.cuda.synchronize()
    assert eng.tables.tolist() == ora.tables and eng.lens.tolist() == ora.lens
    for i, l in enumerate(check_layers):
        assert np.array_equal(u16(eng.k_pool[l]), ora.k_pool[i].view(np.uint16)), f"K layer {l} after set-up"
        assert np.array_equal(u16(eng.v_pool[l]), ora.v_pool[i].view(np.uint16)), f"V layer {l} after set-up"
    for step in range(steps):
        qd, kd, vd = eng.step_inputs(step, "torch")
        out = torch.empty_like(qd)
        eng.step(qd, kd, vd, out)
        torch.cuda.synchronize()
        assert eng.device_status() == 0
        sel = lambda t: t[check_layers].cpu().numpy()
        ref = ora.step(sel(qd), sel(kd), sel(vd), impl="c")
        assert eng.last_slots.tolist() == ora.last_slots
        assert [tuple(p) for p in eng.last_pairs.tolist()] == ora.last_pairs
        assert eng.tables.tolist() == ora.tables
        for i, l in enumerate(check_layers):
            assert np.array_equal(u16(eng.k_pool[l]), ora.k_pool[i].view(np.uint16)), f"K layer {l} step {step}"
            assert_close(out[l].cpu().numpy(), ref[i], f"{w.name} full size, layer {l}, step {step}")
    eng.pool.validate()
    return eng



def test_prefix_full_size_sampled(free_gpu_memory):
    """64 sequences on one 520-token prompt at full size: 63 COW copies in every layer, then decode steps."""
    w = wl.make_workload(3, decode_steps=4)
    eng = _full_size(w, [0, 17, w.num_layers - 1], steps=2)
    assert eng.pool.stats()["cow_copies"] == w.num_seqs - 1


def test_13b_full_size_sampled(free_gpu_memory):
    """13B shape, batch 128, block 32, pool 90 % occupied after churn, full size (40 layers)."""
    w = wl.make_workload(4, decode_steps=4)
    _full_size(w, [0, w.num_layers - 1], steps=2)


@pytest.mark.parametrize("block_size", [256, 8, 64, 512])
def test_long_context_full_size_sampled(block_size, free_gpu_memory):
    """16 sequences of 4k-16k tokens, full size (32 layers): in 4 MiB pages (block 256), and the
    block-size sweep's ends with the same token data -- block 8 gives tables of up to 2049 entries
    (the producer's 128-entry table window is refilled 16 times per (sequence, head)), block 64
    one TMA box per 64-token tile."""
    w = wl.make_workload(5, decode_steps=4, block_size=block_size)
    _full_size(w, [0, w.num_layers - 1], steps=2)


def test_long_context_nhd_full_size_sampled(free_gpu_memory):
    """The long-context workload at full size in NHD pools (block 256: a head's 256-byte row
    every H*D elements), as `bench.py --layout NHD --config 5` runs it; layer 0."""
    w = wl.make_workload(5, decode_steps=4, layout="NHD")
    _full_size(w, [0], steps=1)


def test_early_start_back_to_back_layers():
    """Attention launches flagged to start before their predecessor ends (each follows the previous
    layer's launch, which writes none of its inputs) give the oracle's result on every layer."""
    w = wl.make_workload(2, num_layers=4, num_seqs=8, len_scale=0.3, decode_steps=1)
    eng = DecodeEngine(w, fill="numpy", cascade=False)
    eng.run_script(values="numpy")
    torch.cuda.synchronize()
    q, _, _ = eng.step_inputs(0, "numpy")
    out = torch.full_like(q, float("nan"))
    for rep in range(3):
        for layer in range(w.num_layers):
            eng.attention(layer, q, out, early=rep > 0 or layer > 0)
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    kp, vp = wl.pool_values(w, 0), wl.pool_values(w, 1)
    from oracle import ref_alloc as ra       # the set-up only admits: the oracle allocator's tables
    op = ra.RefPool(w.num_blocks, [int(x) for x in w.free_order])
    tabs = np.asarray([ra.admit(op, int(t), w.block_size, w.max_blocks) for t in w.context_lens], dtype=np.int32)
    lens = np.asarray(w.context_lens, dtype=np.int32)
    assert eng.tables.tolist() == tabs.tolist() and eng.lens.tolist() == lens.tolist()
    for layer in range(w.num_layers):
        ref = rf.decode_attention(q[layer].cpu().numpy(), kp[layer], vp[layer], tabs, lens, w.block_size, w.layout)
        assert_close(out[layer].cpu().numpy(), ref, f"early layer {layer}")


@pytest.mark.parametrize("kv_dtype", ["f16", "e4m3"])
def test_early_start_behind_the_append(kv_dtype):
    """Attention flagged to start early behind the layer's own append launch (the tiles holding
    the appended rows read only after it) writes the same output, bit for bit, as attention
    started after the append, and matches the oracle."""
    w = wl.make_workload(2, num_layers=3, num_seqs=12, len_scale=0.3, decode_steps=2, kv_dtype=kv_dtype)
    eng = DecodeEngine(w, fill="numpy", cascade=False, fused=False)
    ora = make_oracle(w)
    eng.run_script(values="numpy")
    ora.run_script()
    q, k, v = eng.step_inputs(0, "numpy")
    n_slots, n_pairs = eng.prepare_step()
    assert n_slots == w.num_seqs
    if n_pairs:
        eng.pool.copy_blocks(eng.pairs_d, n_pairs, status=eng.status)
    ref = ora.step(*ora.step_inputs(0))
    flags = pkv.binding.ATTN_INPUTS_EARLY | pkv.binding.ATTN_LAST_ROW_PENDING
    outs = []
    for f in (flags, 0):
        out = torch.full_like(q, float("nan"))
        for layer in range(w.num_layers):
            eng.pool.append(layer, k[layer], v[layer], eng.slots_d[:n_slots], status=eng.status)
            eng.pool.decode_attention_ex(layer, q[layer], eng.tables_d, eng.lens_d, out[layer], eng.workspace,
                                         flags=f)
        torch.cuda.synchronize()
        outs.append(out)
    assert eng.device_status() == 0
    assert torch.equal(outs[0], outs[1])
    for layer in range(w.num_layers):
        assert_close(outs[0][layer].cpu().numpy(), ref[layer], f"{kv_dtype} layer {layer}")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_early_start_behind_the_append_edge_lengths(layout):
    """Sequences of 1, 2, 15-17, 63-65 and 300 tokens: the appended row is the first row, the
    last of a block, the first of a new one, alone in its tile or one of many. Attention
    started early behind the append (LAST_ROW_PENDING) equals attention started after it,
    bit for bit, and the oracle on the cache with the rows written in."""
    lens = [1, 2, 15, 16, 17, 63, 64, 65, 300, 1]
    H, D, B = 4, 128, 16
    q, kp, vp, tab, ln, B, N = _raw_case(lens, H=H, D=D, B=B, layout=layout, seed=31)
    rng = np.random.default_rng(32)
    kn = rng.standard_normal((len(lens), H, D)).astype(np.float16)
    vn = rng.standard_normal((len(lens), H, D)).astype(np.float16)
    slots = np.array([tab[s, (t - 1) // B] * B + (t - 1) % B for s, t in enumerate(lens)], dtype=np.int64)
    kp2, vp2 = kp.copy(), vp.copy()
    for s_, sl in enumerate(slots):
        blk, off = sl // B, sl % B
        idx = (blk, off) if layout == "NHD" else (blk, slice(None), off)
        kp2[idx], vp2[idx] = kn[s_], vn[s_]
    ref = rc.decode_attention(q, kp2, vp2, tab, ln, B, layout)
    dev = "cuda"
    outs = []
    for flags in (pkv.binding.ATTN_INPUTS_EARLY | pkv.binding.ATTN_LAST_ROW_PENDING, 0):
        kd, vd = torch.from_numpy(kp[None]).to(dev), torch.from_numpy(vp[None]).to(dev)
        pool = pkv.Pool(1, N, B, H, D, layout, k_pool=kd, v_pool=vd)
        ws = pkv.new_workspace(len(lens), H, D, dev)
        qd, td, ld = (torch.from_numpy(a).to(dev) for a in (q, tab, ln))
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        out = torch.full_like(qd, float("nan"))
        pool.append(0, torch.from_numpy(kn).to(dev), torch.from_numpy(vn).to(dev), torch.from_numpy(slots).to(dev),
                    status=st)
        pool.decode_attention_ex(0, qd, td, ld, out, ws, flags=flags)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and pkv.workspace_status(ws) == 0
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    assert_close(outs[0], ref, f"early behind the append, {layout}")


def test_attention_ex_rejects_unknown_flags():
    w = wl.make_workload(1, decode_steps=1)
    eng = DecodeEngine(w, fill="numpy", cascade=False)
    eng.run_script(values="numpy")
    q, _, _ = eng.step_inputs(0, "numpy")
    with pytest.raises(pkv.binding.PkvError) as e:
        eng.pool.decode_attention_ex(0, q[0], eng.tables_d, eng.lens_d, torch.empty_like(q[0]), eng.workspace,
                                     flags=0x4)
    assert e.value.code == "INVALID_ARG"


def test_launch_info_per_cache_dtype():
    """Persistent grid = CTAs per SM x SMs for both cache types; each variant keeps at least
    the three resident CTAs per SM its register budget is set for."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    f = pkv.decode_launch_info(32, 128, "f16")
    e = pkv.decode_launch_info(32, 128, "e4m3")
    for i in (f, e):
        assert i["num_sms"] == sms and i["grid_ctas"] == i["ctas_per_sm"] * sms and i["ctas_per_sm"] >= 3


def test_wait_limit_flags_timeout_and_context_survives():
    """Failure detection without a fault: a wait that nothing satisfies gives up after its
    limit, flags PKV_DEV_TIMEOUT, and the context keeps working (an attention step after
    it is still right)."""
    from paged_kv_cache_88_gb300 import binding as bd
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.check_wait_limit(st)
    torch.cuda.synchronize()
    assert int(st.item()) & pkv.DEV_TIMEOUT
    w = wl.make_workload(1, decode_steps=1)
    run_parity(w, 1)
