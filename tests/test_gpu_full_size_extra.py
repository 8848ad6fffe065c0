"""Full-size GPU parity of the E4M3 decode step and of the tensor-core prefill, each in the
launch configuration bench.py times, checked against the oracle on sampled outputs.

* E4M3: the engine's default step on the full 7B, forked-prompt, 13B and long-context
  workloads (both layouts for 7B and long); the oracle replays the set-up and the step
  with its own allocator and quantiser from the pools as filled, the codes and scales of
  the checked layers are compared bit for bit, and the attention of the sampled
  sequences (every head) with the float64 definition on code x scale.
* Prefill: the benchmark's causal prefill (whole prompts of the 7B workload; chunks of
  4096 over the long contexts), every row of the sampled (sequence, head) pairs against
  the float64 causal definition, computed on just that sequence's blocks.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_cache_88_gb300.engine import DecodeEngine  # noqa: E402
from oracle import fp8  # noqa: E402
from oracle import ref_attn as rf  # noqa: E402
import workloads as wl  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {np.nanmax(err):.3e}"


@pytest.fixture
def free_gpu_memory():
    yield
    import gc
    gc.collect()
    torch.cuda.empty_cache()


def _sample(lens: np.ndarray, n: int) -> list:
    """The longest, the shortest and evenly spread others (sequence indices)."""
    order = np.argsort(lens, kind="stable")
    pick = {int(order[-1]), int(order[0])}
    for i in np.linspace(0, len(lens) - 1, num=max(n - 2, 0) + 2)[1:-1]:
        pick.add(int(order[int(round(i))]))
    return sorted(pick)


def _e4m3_full(cfg: int, check_layers, n_seqs=None, fused=None, groups=0, cow=0, **kw):
    """The benchmark's E4M3 step (the engine's default: the append inside the attention
    launch while each CTA ends at most four (sequence, head) pairs, else a separate launch)
    at full size, against the oracle on the listed layers: the oracle starts from the pools
    as filled before any write, replays the set-up with its own allocator and quantiser
    (tables, codes and scales bit-exact after it), then takes the step's slots and copies
    from its own allocator, appends with its own quantiser (codes and scales bit-exact
    again) and computes the attention of the sampled sequences (every head). ``fused`` is
    the choice the engine must make here, ``cow`` the set-up's copies, ``groups`` the
    cascade's groups."""
    import dataclasses
    from oracle.driver import OracleEngine
    w = wl.make_workload(cfg, kv_dtype="e4m3", **kw)
    eng = DecodeEngine(w, fill="torch")
    assert eng.fused == fused
    snap = [np.stack([t[l].cpu().numpy() for l in check_layers])
            for t in (eng.k_pool, eng.v_pool, eng.k_scale, eng.v_scale)]
    eng.run_script(values="torch")
    assert eng.pool.stats()["cow_copies"] == cow
    ora = OracleEngine(dataclasses.replace(w, num_layers=len(check_layers)), *snap)
    del snap

    def values(op_index, i, which, n):
        return wl.torch_normal_fp16(w.seed, (400 + which, op_index, check_layers[i]), (n, w.num_heads, w.head_dim),
                                    "cuda").cpu().numpy()

    ora.run_script(values)
    torch.cuda.synchronize()
    assert eng.tables.tolist() == ora.tables and eng.lens.tolist() == ora.lens

    def same_pools(what):
        for i, l in enumerate(check_layers):
            assert np.array_equal(eng.k_pool[l].cpu().numpy(), ora.k_pool[i]), f"K codes layer {l} {what}"
            assert np.array_equal(eng.v_pool[l].cpu().numpy(), ora.v_pool[i]), f"V codes layer {l} {what}"
            assert np.array_equal(eng.k_scale[l].cpu().numpy().view(np.uint32), ora.k_scale[i].view(np.uint32)), \
                f"K scales layer {l} {what}"
            assert np.array_equal(eng.v_scale[l].cpu().numpy().view(np.uint32), ora.v_scale[i].view(np.uint32)), \
                f"V scales layer {l} {what}"

    same_pools("after set-up")
    qd, kd, vd = eng.step_inputs(0, "torch")
    out = torch.empty_like(qd)
    eng.step(qd, kd, vd, out)
    torch.cuda.synchronize()
    assert eng.device_status() == 0
    assert eng.plan_groups == groups
    slots, pairs = ora.pool.prepare_append(ora.tables, ora.lens, [1] * w.num_seqs, w.block_size, w.max_blocks)
    assert eng.last_slots.tolist() == slots and [tuple(p) for p in eng.last_pairs.tolist()] == pairs
    assert eng.tables.tolist() == ora.tables
    ora._copy(pairs)
    for i, l in enumerate(check_layers):
        fp8.append_kv(ora.k_pool[i], ora.v_pool[i], ora.k_scale[i], ora.v_scale[i], kd[l].cpu().numpy(),
                      vd[l].cpu().numpy(), slots, w.block_size, w.layout)
    same_pools("after the step's append")
    tab, lens = ora.tables_array(), np.asarray(ora.lens, dtype=np.int32)
    seqs = list(range(w.num_seqs)) if n_seqs is None else _sample(lens, n_seqs)
    for i, l in enumerate(check_layers):
        q = qd[l].cpu().numpy()[seqs]
        ref = fp8.decode_attention(q, ora.k_pool[i], ora.v_pool[i], ora.k_scale[i], ora.v_scale[i], tab[seqs],
                                   lens[seqs], w.block_size, layout=w.layout)
        assert_close(out[l].cpu().numpy()[seqs], ref, f"E4M3 cfg {cfg} layer {l}")


def test_e4m3_7b_full_size_sampled(free_gpu_memory):
    """7B shape, batch 32, 32 layers: layers 0 and 31, every sequence and head."""
    _e4m3_full(2, [0, 31], fused=True)


def test_e4m3_long_context_full_size_sampled(free_gpu_memory):
    """16 sequences of 4k-16k tokens, block 256: layer 0, four sequences, every head."""
    _e4m3_full(5, [0], n_seqs=4, fused=True)


def test_e4m3_prefix_cow_cascade_full_size_sampled(free_gpu_memory):
    """Forked prompt at full size with an E4M3 cache (64 sequences on one 520-token prompt,
    32 layers, codes and scales copied on write for 63 of them in the set-up): the cascade's
    prefix pass over the shared 512 tokens and the private pass with the append inside;
    layers 0 and 31, eight sequences, every head."""
    _e4m3_full(3, [0, 31], n_seqs=8, fused=True, groups=1, cow=63)


def test_e4m3_nhd_full_size_sampled(free_gpu_memory):
    """E4M3 codes in NHD pools (a head's 128-byte row every H*D bytes; scales [N][H][B] as in
    HND), as `bench.py --kv-dtype e4m3 --layout NHD` runs them: the 7B workload (layers 0 and
    31, every sequence and head) and the long one (layer 0, four sequences)."""
    _e4m3_full(2, [0, 31], fused=True, layout="NHD")
    _e4m3_full(5, [0], n_seqs=4, fused=True, layout="NHD")


def test_e4m3_13b_full_size_sampled(free_gpu_memory):
    """13B shape, batch 128, block 32, pool 90 % occupied after churn, 40 layers (the tensor-core
    E4M3 consumer at its largest batch): layers 0 and 39, sixteen sequences, every head."""
    _e4m3_full(4, [0, 39], n_seqs=16, fused=False)


def test_e4m3_long_context_block_16_full_size_sampled(free_gpu_memory):
    """The long-context workload at block 16 (four TMA boxes per 64-token tile, 128-entry table
    windows refilled along 16k-token sequences): layer 0, four sequences, every head."""
    _e4m3_full(5, [0], n_seqs=4, block_size=16, fused=True)


@pytest.mark.parametrize("block_size", [64, 512])
def test_e4m3_long_context_block_sweep_full_size_sampled(block_size, free_gpu_memory):
    """The long-context E4M3 rows of the block-size sweep at full size (block 64: one TMA box
    a tile; block 512: the quantised cache's 512-token pages): layer 0, two sequences."""
    _e4m3_full(5, [0], n_seqs=2, block_size=block_size, fused=True)


def _prefill_full(cfg: int, chunk: int, n_seqs: int, heads, block_size=None):
    w = wl.make_workload(cfg, decode_steps=8, block_size=block_size)
    eng = DecodeEngine(w, fill="torch")
    eng.run_script(values="torch")
    H, D, B = w.num_heads, w.head_dim, w.block_size
    # the set-up only admits sequences (the pools keep their generated values): the oracle
    # allocator's tables for the same admissions, equal to the library's
    from oracle import ref_alloc as ra
    op = ra.RefPool(w.num_blocks, [int(x) for x in w.free_order])
    tabs = np.asarray([ra.admit(op, int(t), B, w.max_blocks) for t in w.context_lens], dtype=np.int64)
    lens = np.asarray(w.context_lens, dtype=np.int64)
    assert eng.tables.tolist() == tabs.tolist() and eng.lens.tolist() == lens.tolist()
    chunks = np.minimum(lens, chunk).astype(np.int64)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + cfg)
    q = torch.randn((int(q_start[-1]), H, D), generator=g, device="cuda").to(torch.float16)
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eng.pool.prefill_attention(0, q, torch.from_numpy(q_start).cuda(), int(chunks.max()), eng.tables_d, eng.lens_d,
                               out, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for s in _sample(lens, n_seqs):
        T, C = int(lens[s]), int(chunks[s])
        nb = -(-T // B)
        blocks = torch.from_numpy(tabs[s, :nb]).cuda()
        tab = np.arange(nb, dtype=np.int32)[None]
        r0, r1 = int(q_start[s]), int(q_start[s + 1])
        for h in heads:
            kp = eng.k_pool[0][blocks][:, h:h + 1].cpu().numpy()        # [nb, 1, B, D]: this head's blocks
            vp = eng.v_pool[0][blocks][:, h:h + 1].cpu().numpy()
            qs = q[r0:r1, h:h + 1].cpu().numpy()
            ref = rf.prefill_attention(qs, kp, vp, tab, [T], [0, C], B, layout="HND")
            assert_close(out[r0:r1, h:h + 1].cpu().numpy(), ref, f"prefill cfg {cfg} seq {s} head {h}")


def test_prefill_whole_prompts_7b_full_size_sampled(free_gpu_memory):
    """The benchmark's whole-prompt prefill (chunks of up to 2048) on the 7B workload:
    four sequences, heads 0 and 31, every row."""
    _prefill_full(2, 2048, 4, [0, 31])


def test_prefill_chunks_of_512_7b_full_size_sampled(free_gpu_memory):
    """The benchmark's 7B prefill in chunks of 512 (each sequence's last 512 tokens over the
    rest of its context): four sequences, heads 0 and 31, every row."""
    _prefill_full(2, 512, 4, [0, 31])


@pytest.mark.parametrize("block_size", [16, 512])
def test_prefill_long_chunks_other_blocks_full_size_sampled(block_size, free_gpu_memory):
    """The 4096-token chunks over the long contexts at blocks 16 and 512 (the prefill rows of
    the block-size sweep): the longest and the shortest sequence, head 0, every row."""
    _prefill_full(5, 4096, 2, [0], block_size=block_size)


def test_prefill_long_chunks_full_size_sampled(free_gpu_memory):
    """The benchmark's 4096-token chunks over the long contexts (block 256): the longest and
    the shortest sequence, heads 0 and 17, every row."""
    _prefill_full(5, 4096, 2, [0, 17])
