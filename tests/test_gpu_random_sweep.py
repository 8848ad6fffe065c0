"""Seeded random sweep of the decode step's GPU path against the oracle.

Each case draws the batch size, heads, head_dim, block size, layout and a length mix
that hits the edges (a context of only the appended token, a block or a 64-token tile
boundary on either side, long contexts), scatters the blocks over a shuffled pool whose
unused rows (and, before the append, the appended ones) hold NaN, appends one token per
sequence through pkv_append (quantising on an E4M3 pool) and attends with
pkv_decode_attention_ex, with or without the early start behind the append (a read of an
appended row before the append lands would bring in a NaN or a stale code). The pools
after the append (codes and scales on E4M3) must equal the oracle's bit for bit, and the
attention must match the float64 oracle within the decode tolerance.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_88_gb300 as pkv  # noqa: E402
from paged_kv_cache_88_gb300 import binding as bd  # noqa: E402
from oracle import fp8  # noqa: E402
from oracle import ref_attn_c as rc  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2
BLOCK_SIZES = [8, 16, 32, 64, 128, 256, 512]


def assert_close(got, ref, what):
    err = np.abs(got.astype(np.float64) - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {np.nanmax(err):.3e}"


def draw_lengths(rng, S, B, long_max):
    """Lengths after the append (each >= 1: the appended token is the last row)."""
    edges = [1, 2, B - 1, B, B + 1, 2 * B, 2 * B + 1, 63, 64, 65, 127, 128, 129]
    out = []
    for _ in range(S):
        r = rng.random()
        if r < 0.5:
            out.append(int(rng.choice([e for e in edges if e >= 1])))
        else:
            out.append(int(rng.integers(1, long_max + 1)))
    return out


def draw_tables(rng, lens, B, spare=3):
    nb = [-(-t // B) for t in lens]
    N = sum(nb) + spare
    perm = rng.permutation(N).astype(np.int32)
    maxb = max(nb)
    tables = np.zeros((len(lens), maxb), dtype=np.int32)
    i = 0
    for s, n in enumerate(nb):
        tables[s, :n] = perm[i:i + n]
        i += n
    return tables, N


def slots_of(tables, lens, B):
    return np.array([tables[s, (t - 1) // B] * B + (t - 1) % B for s, t in enumerate(lens)], dtype=np.int64)


CASES = list(range(40))


@pytest.mark.parametrize("case", CASES)
def test_random_fp16_step(case):
    rng = np.random.default_rng(7000 + case)
    S = int(rng.integers(1, 41))
    H = int(rng.choice([1, 2, 3, 4, 8]))
    D = int(rng.choice([64, 128, 256]))
    B = int(rng.choice(BLOCK_SIZES))
    layout = str(rng.choice(["NHD", "HND"]))
    flags = int(rng.choice([0, bd.ATTN_INPUTS_EARLY | bd.ATTN_LAST_ROW_PENDING]))
    lens = draw_lengths(rng, S, B, long_max=2000 if D < 256 else 1000)
    tables, N = draw_tables(rng, lens, B)
    shape = (N, B, H, D) if layout == "NHD" else (N, H, B, D)
    kp = np.full(shape, np.uint16(0x7E00), dtype=np.uint16).view(np.float16)   # NaN outside the contexts
    vp = kp.copy()
    for s, t in enumerate(lens):
        for tok in range(t - 1):                                              # the last row is appended
            blk, off = tables[s, tok // B], tok % B
            idx = (blk, off) if layout == "NHD" else (blk, slice(None), off)
            kp[idx] = rng.standard_normal((H, D)).astype(np.float16)
            vp[idx] = rng.standard_normal((H, D)).astype(np.float16)
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    kn = rng.standard_normal((S, H, D)).astype(np.float16)
    vn = rng.standard_normal((S, H, D)).astype(np.float16)
    slots = slots_of(tables, lens, B)
    # the oracle's cache: the appended rows written in
    kr, vr = kp.copy(), vp.copy()
    for s, sl in enumerate(slots):
        blk, off = sl // B, sl % B
        idx = (blk, off) if layout == "NHD" else (blk, slice(None), off)
        kr[idx], vr[idx] = kn[s], vn[s]
    ln = np.asarray(lens, dtype=np.int32)
    ref = rc.decode_attention(q, kr, vr, tables, ln, B, layout)

    dev = "cuda"
    kd, vd = torch.from_numpy(kp[None]).to(dev), torch.from_numpy(vp[None]).to(dev)
    pool = pkv.Pool(1, N, B, H, D, layout, k_pool=kd, v_pool=vd)
    ws = pkv.new_workspace(S, H, D, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    qd, td, ld = (torch.from_numpy(a).to(dev) for a in (q, tables, ln))
    out = torch.full_like(qd, float("nan"))
    pool.append(0, torch.from_numpy(kn).to(dev), torch.from_numpy(vn).to(dev), torch.from_numpy(slots).to(dev),
                status=st)
    pool.decode_attention_ex(0, qd, td, ld, out, ws, flags=flags)
    torch.cuda.synchronize()
    what = f"case {case}: S={S} H={H} D={D} B={B} {layout} flags={flags}"
    assert int(st.item()) == 0 and pkv.workspace_status(ws) == 0, what
    assert np.array_equal(kd[0].cpu().numpy().view(np.uint16), kr.view(np.uint16)), what
    assert np.array_equal(vd[0].cpu().numpy().view(np.uint16), vr.view(np.uint16)), what
    assert_close(out.cpu().numpy(), ref, what)


@pytest.mark.parametrize("case", CASES[:24])
def test_random_e4m3_step(case):
    rng = np.random.default_rng(8000 + case)
    S = int(rng.integers(1, 13))
    H = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([64, 128]))
    B = int(rng.choice(BLOCK_SIZES))
    flags = int(rng.choice([0, bd.ATTN_INPUTS_EARLY | bd.ATTN_LAST_ROW_PENDING]))
    layout = str(rng.choice(["NHD", "HND"]))
    lens = draw_lengths(rng, S, B, long_max=700)
    tables, N = draw_tables(rng, lens, B)
    kc = rng.integers(0, 256, size=(N, H, B, D), dtype=np.uint8)          # made HND, turned NHD below
    vc = rng.integers(0, 256, size=(N, H, B, D), dtype=np.uint8)
    for c_ in (kc, vc):
        c_[(c_ & 0x7F) == 0x7F] ^= 1                      # no NaN code inside a context
    ks = rng.uniform(0.001, 0.01, size=(N, H, B)).astype(np.float32)
    vs = rng.uniform(0.001, 0.01, size=(N, H, B)).astype(np.float32)
    live = np.zeros((N, B), dtype=bool)
    for s, t in enumerate(lens):
        for tok in range(t):
            live[tables[s, tok // B], tok % B] = True
    dead = ~live
    kc.transpose(0, 2, 1, 3)[dead] = 0x7F                    # NaN codes and scales past every context
    vc.transpose(0, 2, 1, 3)[dead] = 0xFF
    ks.transpose(0, 2, 1)[dead] = np.nan
    vs.transpose(0, 2, 1)[dead] = np.nan
    if layout == "NHD":
        kc, vc = np.ascontiguousarray(kc.transpose(0, 2, 1, 3)), np.ascontiguousarray(vc.transpose(0, 2, 1, 3))
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    kn = rng.standard_normal((S, H, D)).astype(np.float16)
    vn = rng.standard_normal((S, H, D)).astype(np.float16)
    slots = slots_of(tables, lens, B)
    kcr, vcr, ksr, vsr = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    fp8.append_kv(kcr, vcr, ksr, vsr, kn, vn, slots, B, layout=layout)
    ln = np.asarray(lens, dtype=np.int32)
    ref = fp8.decode_attention(q, kcr, vcr, ksr, vsr, tables, ln, B, layout=layout)

    dev = "cuda"
    kd, vd = torch.from_numpy(kc[None]).to(dev), torch.from_numpy(vc[None]).to(dev)
    ksd, vsd = torch.from_numpy(ks[None]).to(dev), torch.from_numpy(vs[None]).to(dev)
    pool = pkv.Pool(1, N, B, H, D, layout, k_pool=kd, v_pool=vd, kv_dtype="e4m3", k_scale=ksd, v_scale=vsd)
    ws = pkv.new_workspace(S, H, D, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    qd, td, ld = (torch.from_numpy(a).to(dev) for a in (q, tables, ln))
    out = torch.full_like(qd, float("nan"))
    pool.append(0, torch.from_numpy(kn).to(dev), torch.from_numpy(vn).to(dev), torch.from_numpy(slots).to(dev),
                status=st)
    pool.decode_attention_ex(0, qd, td, ld, out, ws, flags=flags)
    torch.cuda.synchronize()
    what = f"case {case}: S={S} H={H} D={D} B={B} {layout} flags={flags}"
    assert int(st.item()) == 0 and pkv.workspace_status(ws) == 0, what
    assert np.array_equal(kd[0].cpu().numpy(), kcr) and np.array_equal(vd[0].cpu().numpy(), vcr), what
    assert np.array_equal(ksd[0].cpu().numpy().view(np.uint32), ksr.view(np.uint32)), what
    assert np.array_equal(vsd[0].cpu().numpy().view(np.uint32), vsr.view(np.uint32)), what
    assert_close(out.cpu().numpy(), ref, what)


def random_fork_spec(rng, B, max_prefix=2048):
    """Groups of sequences forked from a root (sharing its first nsh full blocks, then
    private tails of 0 to 5 blocks, some ending exactly at the prefix), plus unshared
    sequences; in the (s, ...) form of the cascade tests' builders."""
    spec = []
    for _ in range(int(rng.integers(1, 4))):
        nsh = int(rng.integers(1, max_prefix // B + 2))
        root = len(spec)
        spec.append((None, 0, nsh * B + int(rng.integers(0, 3 * B))))
        for _ in range(int(rng.integers(1, 30))):
            spec.append((root, nsh, nsh * B + int(rng.integers(0, 5 * B))))
    for _ in range(int(rng.integers(0, 4))):
        spec.append((None, 0, int(rng.integers(1, 600))))
    return spec


@pytest.mark.parametrize("case", CASES[:12])
def test_random_fp16_cascade(case):
    """The planned cascade (prefix pass, then the private pass merging its pieces) on random
    fork structures equals the plain float64 attention."""
    from tests.test_gpu_cascade import Case
    rng = np.random.default_rng(9000 + case)
    B = int(rng.choice(BLOCK_SIZES))
    H = int(rng.choice([1, 2, 4]))
    c = Case(random_fork_spec(rng, B), H=H, B=B, seed=9100 + case)
    groups, begin = c.plan()
    ref = c.oracle()
    what = f"case {case}: S={c.S} H={H} B={B} groups={len(groups)}"
    if len(groups):
        splits = bd.prefix_splits(len(groups), H, int(groups[:, 2].max()))
        c.prefix(groups, splits)
        got = c.decode(begin, splits)
    else:
        got = c.decode(None, 0)
    assert int(c.status.item()) == 0 and bd.workspace_status(c.ws) == 0, what
    assert_close(got, ref, what)


@pytest.mark.parametrize("case", CASES[:8])
def test_random_e4m3_cascade(case):
    from tests.test_gpu_cascade_e4m3 import Q8Case
    rng = np.random.default_rng(9500 + case)
    B = int(rng.choice(BLOCK_SIZES))
    H = int(rng.choice([1, 2, 4]))
    c = Q8Case(random_fork_spec(rng, B, max_prefix=768), H=H, B=B, seed=9600 + case)
    groups, begin = c.plan()
    ref = c.oracle()
    what = f"case {case}: S={c.S} H={H} B={B} groups={len(groups)}"
    if len(groups):
        splits = bd.prefix_splits(len(groups), H, int(groups[:, 2].max()))
        c.prefix(groups, splits)
        got = c.decode(begin, splits)
    else:
        got = c.decode(None, 0)
    assert int(c.status.item()) == 0 and bd.workspace_status(c.ws) == 0, what
    assert_close(got, ref, what)


@pytest.mark.parametrize("case", CASES[:16])
def test_random_prefill(case):
    """Paged causal prefill of random chunks (the last c tokens of each context, c from 1 to
    the whole context; chunk and context lengths on tile boundaries and between) over
    NaN-guarded pools of every block size, against the float64 prefill definition."""
    from oracle import ref_attn as rf
    from tests.test_gpu_prefill import _case, _run, _check
    rng = np.random.default_rng(9900 + case)
    B = int(rng.choice(BLOCK_SIZES))
    H = int(rng.choice([1, 2, 3]))
    S = int(rng.integers(1, 9))
    edges = [1, 2, 127, 128, 129, 255, 256, 257, 383, 384, 511, 512]
    lens, chunks = [], []
    for _ in range(S):
        T = int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 1600))
        c = int(rng.choice([e for e in edges if e <= T] + [T])) if rng.random() < 0.5 else int(rng.integers(1, T + 1))
        lens.append(T)
        chunks.append(min(c, T))
    q, qs, kp, vp, tab, ln, N = _case(lens, chunks, H, B, seed=9950 + case)
    got, st = _run(q, qs, kp, vp, tab, ln, N, H, B, max(chunks))
    what = f"case {case}: B={B} H={H} lens={lens} chunks={chunks}"
    assert st == 0, what
    _check(got, rf.prefill_attention(q, kp, vp, tab, ln, qs, B, layout="HND"), what)
