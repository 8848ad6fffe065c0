"""GPU parity of the shared-prefix (cascade) decode against the oracle.

The prefix pass (pkv_prefix_attention) is checked piece by piece: o / l is the
softmax-weighted mean of V over the piece's keys and m + log2(l) is
log2 sum_t 2^(scale log2(e) q.K_t) over them, both in float64 on the host. The
whole cascade (prefix pass, then pkv_decode_attention_ex) is checked against
the plain float64 attention of the oracle; so is the engine's decode step with
the cascade on, on the forked-prompt workload.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import paged_kv_cache_88_gb300 as pkv  # noqa: E402
from paged_kv_cache_88_gb300 import binding as bd  # noqa: E402
from oracle import ref_attn as rf  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2
D = 128
LOG2E = 1.4426950408889634


def assert_close(got, ref, what, atol=ATOL, rtol=RTOL):
    err = np.abs(got.astype(np.float64) - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {np.nanmax(err):.3e}"


def build_case(spec, H, B, seed):
    """spec: list of (shared_with, shared_blocks, T): sequence s copies the first
    shared_blocks ids of sequence shared_with (or shares none), then gets fresh
    blocks up to T tokens. Slots past each context hold NaN."""
    rng = np.random.default_rng(seed)
    S = len(spec)
    maxb = max(-(-T // B) for _, _, T in spec)
    tables = np.full((S, maxb), -1, dtype=np.int32)
    nxt = 0
    for s, (src, nsh, T) in enumerate(spec):
        nb = -(-T // B)
        if src is not None:
            tables[s, :nsh] = tables[src, :nsh]
        else:
            nsh = 0
        tables[s, nsh:nb] = np.arange(nxt, nxt + nb - nsh)
        nxt += nb - nsh
    N = nxt + 2
    perm = rng.permutation(N).astype(np.int32)     # scatter the blocks over the pool
    tables = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    lens = np.array([T for _, _, T in spec], dtype=np.int32)
    kp = rng.standard_normal((N, H, B, D)).astype(np.float16)
    vp = rng.standard_normal((N, H, B, D)).astype(np.float16)
    for s, T in enumerate(lens):
        nb = -(-int(T) // B)
        off = int(T) - (nb - 1) * B
        if off < B:
            kp[tables[s, nb - 1], :, off:] = np.float16(np.nan)
            vp[tables[s, nb - 1], :, off:] = np.float16(np.nan)
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    return q, kp, vp, tables, lens, N


class Case:
    def __init__(self, spec, H=4, B=16, seed=0, scale=0.0):
        self.q, self.kp, self.vp, self.tables, self.lens, self.N = build_case(spec, H, B, seed)
        self.H, self.B, self.S = H, B, len(spec)
        self.scale = scale if scale > 0 else 1.0 / math.sqrt(D)
        dev = "cuda"
        self.pool = pkv.Pool(1, self.N, B, H, D, "HND", k_pool=torch.from_numpy(self.kp).to(dev),
                             v_pool=torch.from_numpy(self.vp).to(dev))
        self.qd = torch.from_numpy(self.q).to(dev)
        self.tab_d = torch.from_numpy(self.tables).to(dev)
        self.lens_d = torch.from_numpy(self.lens).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pieces = torch.full((bd.prefix_pieces_bytes(self.S, H, D) // 4,), float("nan"), device=dev)
        self.ws = bd.new_workspace(self.S, H, D)

    def plan(self, **kw):
        g, b = bd.cascade_plan(self.tables, self.lens, self.B, **kw)
        return g.copy(), b.copy()

    def prefix(self, groups, splits, scale=0.0):
        gd = torch.from_numpy(np.ascontiguousarray(groups, dtype=np.int32)).cuda()
        self.pool.prefix_attention(0, self.qd, gd, len(groups), splits, self.tab_d, self.pieces, self.status,
                                   scale=scale)

    def decode(self, begin, splits, scale=0.0, **kw):
        out = torch.full_like(self.qd, float("nan"))
        bdv = torch.from_numpy(np.ascontiguousarray(begin, dtype=np.int32)).cuda() if begin is not None else None
        self.pool.decode_attention_ex(0, self.qd, self.tab_d, self.lens_d, out, self.ws, seq_begin=bdv,
                                      pieces=self.pieces if begin is not None else None, splits=splits,
                                      scale=scale, **kw)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def oracle(self):
        return rf.decode_attention(self.q, self.kp, self.vp, self.tables, self.lens, self.B, layout="HND",
                                   scale=self.scale)

    def keys(self, s, h, t0, t1):
        k = rf.gather_sequence(self.kp, self.tables[s], t1, h, "HND", self.H, self.B, D)[t0:]
        v = rf.gather_sequence(self.vp, self.tables[s], t1, h, "HND", self.H, self.B, D)[t0:]
        return k, v


def forked_spec(n, shared_blocks, suffix, B, rng):
    spec = [(None, 0, shared_blocks * B + int(rng.integers(1, suffix)))]
    spec += [(0, shared_blocks, shared_blocks * B + int(rng.integers(1, suffix))) for _ in range(n - 1)]
    return spec


@pytest.mark.parametrize("splits", [1, 2, 3, 8])
def test_prefix_pieces(splits):
    """Each piece against its keys: a ragged last key tile (P = 1040), and splits with no keys."""
    rng = np.random.default_rng(1)
    B = 16
    spec = forked_spec(5, 65, 40, B, rng) + [(None, 0, 300)] + forked_spec(3, 4, 100, B, rng)
    spec[6:] = [(6, 4, T) if src is not None else (None, 0, T) for src, _, T in spec[6:]]
    c = Case(spec, H=3, B=B, seed=2)
    groups, begin = c.plan()
    assert groups[:, :3].tolist() == [[0, 5, 1040], [6, 3, 64]]
    c.prefix(groups, splits)
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    pcs = c.pieces.cpu().numpy().reshape(c.S, c.H, bd.MAX_PREFIX_SPLITS, D + 4)
    sl2 = c.scale * LOG2E
    for f, n, P, _ in groups.tolist():
        per = -(-(-(-P // 128)) // splits) * 128
        for s in range(f, f + n):
            for h in range(c.H):
                for k in range(splits):
                    t0, t1 = min(P, k * per), min(P, (k + 1) * per)
                    o, m, l = pcs[s, h, k, :D], pcs[s, h, k, D], pcs[s, h, k, D + 1]
                    if t0 >= t1:
                        assert m == -np.inf and l == 0 and not o.any(), (s, h, k)
                        continue
                    kk, vv = c.keys(s, h, t0, t1)
                    x = sl2 * (kk @ c.q[s, h].astype(np.float64))
                    lse2 = x.max() + math.log2(np.exp2(x - x.max()).sum())
                    assert abs(float(m) + math.log2(float(l)) - lse2) < 3e-3, (s, h, k)
                    assert float(m) >= x.max() - 8.0 - 1e-3
                    assert_close(o / l, rf.attend(c.q[s, h], kk, vv, c.scale), f"piece {(s, h, k)}")


@pytest.mark.parametrize("splits", [1, 3])
def test_prefix_pieces_early_start_identical(splits):
    """Started early behind a preceding attention launch, the prefix pass writes the same
    pieces, bit for bit, as started after it (and over pieces that launch left as NaN)."""
    rng = np.random.default_rng(3)
    B = 16
    spec = forked_spec(6, 40, 60, B, rng) + forked_spec(4, 9, 30, B, rng)
    spec[6:] = [(6, 9, T) if src is not None else (None, 0, T) for src, _, T in spec[6:]]
    c = Case(spec, H=4, B=B, seed=4)
    groups, begin = c.plan()
    assert groups[:, :3].tolist() == [[0, 6, 640], [6, 4, 144]]
    c.prefix(groups, splits)
    torch.cuda.synchronize()
    ref = c.pieces.clone()
    gd = torch.from_numpy(np.ascontiguousarray(groups, dtype=np.int32)).cuda()
    for _ in range(2):
        c.pieces.fill_(float("nan"))
        # a preceding kernel on the stream, then the prefix pass that may start before it ends
        c.pool.decode_attention_ex(0, c.qd, c.tab_d, c.lens_d, torch.empty_like(c.qd), c.ws)
        c.pool.prefix_attention(0, c.qd, gd, len(groups), splits, c.tab_d, c.pieces, c.status,
                                flags=bd.ATTN_INPUTS_EARLY)
        torch.cuda.synchronize()
        assert int(c.status.item()) == 0
        for f, n, _, _ in groups.tolist():
            got = c.pieces.view(c.S, c.H, bd.MAX_PREFIX_SPLITS, D + 4)[f:f + n, :, :splits]
            want = ref.view(c.S, c.H, bd.MAX_PREFIX_SPLITS, D + 4)[f:f + n, :, :splits]
            assert torch.equal(got, want)


@pytest.mark.parametrize("B", [8, 16, 64, 256, 512])
def test_cascade_matches_oracle(B):
    """Two groups, unshared sequences, and a member whose whole context is the prefix."""
    rng = np.random.default_rng(B)
    nsh = max(1, 600 // B)
    spec = forked_spec(6, nsh, 3 * B, B, rng)
    spec += [(None, 0, int(rng.integers(1, 700))), (None, 0, 5)]
    g2 = len(spec)
    spec += [(None, 0, 2 * B + 7), (g2, 2, 2 * B + 3), (g2, 2, 2 * B)]     # the last: no private tokens
    c = Case(spec, H=4, B=B, seed=B + 1)
    groups, begin = c.plan()
    assert len(groups) == 2 and begin[-1] == c.lens[-1]
    splits = bd.prefix_splits(len(groups), c.H, int(groups[:, 2].max()))
    c.prefix(groups, splits)
    got = c.decode(begin, splits)
    assert int(c.status.item()) == 0 and bd.workspace_status(c.ws) == 0
    assert_close(got, c.oracle(), f"cascade B={B}")
    # the same call without the cascade
    assert_close(c.decode(None, 0), c.oracle(), f"plain B={B}")


def test_cascade_explicit_scale_and_forced_splits():
    rng = np.random.default_rng(7)
    c = Case(forked_spec(9, 40, 50, 16, rng), H=2, B=16, seed=8, scale=0.2)
    groups, begin = c.plan()
    for splits in (1, 5, 8):
        c.prefix(groups, splits, scale=0.2)
        assert_close(c.decode(begin, splits, scale=0.2), c.oracle(), f"splits {splits}")


def test_cascade_with_fused_append():
    """One decode step: the new token appended inside the private pass, attention over it."""
    rng = np.random.default_rng(11)
    B, H = 16, 4
    spec = forked_spec(7, 20, 30, B, rng)
    c = Case(spec, H=H, B=B, seed=12)
    # the new token goes to the slot of position T_s - 1: the context already counts it
    slots = np.array([int(c.tables[s, (T - 1) // B]) * B + (T - 1) % B for s, T in enumerate(c.lens)],
                     dtype=np.int64)
    kn = rng.standard_normal((c.S, H, D)).astype(np.float16)
    vn = rng.standard_normal((c.S, H, D)).astype(np.float16)
    groups, begin = c.plan()
    assert len(groups) == 1 and (begin == 320).all()
    c.prefix(groups, 2)
    got = c.decode(begin, 2, k_new=torch.from_numpy(kn).cuda(), v_new=torch.from_numpy(vn).cuda(),
                   slot_mapping=torch.from_numpy(slots).cuda())
    rf.append_kv(c.kp, c.vp, kn, vn, slots, B, "HND")
    assert_close(got, c.oracle(), "cascade + append")
    assert np.array_equal(c.pool.k_pool.cpu().numpy().reshape(-1).view(np.uint16), c.kp.reshape(-1).view(np.uint16))


def test_bad_begin_is_flagged_and_attends_everything():
    rng = np.random.default_rng(5)
    c = Case(forked_spec(4, 10, 40, 16, rng), H=2, B=16, seed=6)
    groups, begin = c.plan()
    c.prefix(groups, 1)
    begin = begin.copy()
    begin[1] = 17                       # not whole blocks: read as 0, the whole context attended here
    got = c.decode(begin, 1)
    assert bd.workspace_status(c.ws) & 0x2
    assert_close(got, c.oracle(), "bad begin")


def test_cascade_argument_errors():
    rng = np.random.default_rng(9)
    c = Case(forked_spec(3, 10, 20, 16, rng), H=2, B=16, seed=10)
    groups, begin = c.plan()
    gd = torch.from_numpy(groups).cuda()
    for splits in (0, bd.MAX_PREFIX_SPLITS + 1):
        with pytest.raises(bd.PkvError) as e:
            c.pool.prefix_attention(0, c.qd, gd, len(groups), splits, c.tab_d, c.pieces, c.status)
        assert e.value.code == "INVALID_ARG"
    with pytest.raises(bd.PkvError) as e:    # pieces too small
        c.pool.prefix_attention(0, c.qd, gd, len(groups), 1, c.tab_d, c.pieces[:16], c.status)
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(bd.PkvError) as e:    # an unknown flag bit
        c.pool.prefix_attention(0, c.qd, gd, len(groups), 1, c.tab_d, c.pieces, c.status, flags=0x2)
    assert e.value.code == "INVALID_ARG"
    with pytest.raises(bd.PkvError) as e:    # seq_begin without pieces
        c.pool.decode_attention_ex(0, c.qd, c.tab_d, c.lens_d, torch.empty_like(c.qd), c.ws,
                                   seq_begin=torch.from_numpy(begin).cuda(), splits=1)
    assert e.value.code == "INVALID_ARG"
    # an fp16 pool with head_dim 64 has no prefix pass
    small = pkv.Pool(1, 8, 16, 2, 64, "HND", k_pool=torch.zeros((8, 2, 16, 64), dtype=torch.float16, device="cuda"),
                     v_pool=torch.zeros((8, 2, 16, 64), dtype=torch.float16, device="cuda"))
    with pytest.raises(bd.PkvError) as e:
        small.prefix_attention(0, torch.zeros((3, 2, 64), dtype=torch.float16, device="cuda"), gd, 1, 1, c.tab_d,
                               c.pieces, c.status)
    assert e.value.code == "UNSUPPORTED"
    # nor has an NHD pool, fp16 or E4M3 (a head's rows are not contiguous there)
    for kv in ("f16", "e4m3"):
        dt = torch.float16 if kv == "f16" else torch.uint8
        nhd = pkv.Pool(1, 8, 16, 2, 128, "NHD", kv_dtype=kv, k_pool=torch.zeros((8, 16, 2, 128), dtype=dt, device="cuda"),
                       v_pool=torch.zeros((8, 16, 2, 128), dtype=dt, device="cuda"))
        with pytest.raises(bd.PkvError) as e:
            nhd.prefix_attention(0, torch.zeros((3, 2, 128), dtype=torch.float16, device="cuda"), gd, 1, 1, c.tab_d,
                                 c.pieces, c.status)
        assert e.value.code == "UNSUPPORTED"
    torch.cuda.synchronize()


@pytest.mark.parametrize("splits", [1, 3, 8])
def test_merge_of_given_pieces(splits):
    """pkv_decode_attention_ex merges whatever prefix pieces it is given: pieces written
    here (random m, l and o, one of them empty), private contexts of every kind (several
    tiles, one token, none at all, no cascade for the sequence). Expected: the float64
    merge of the pieces with the softmax sums of the private keys."""
    hd = 128
    rng = np.random.default_rng(hd * 10 + splits)
    H, B = 3, 16
    lens = np.array([300, 41, 16, 128, 70, 200, 1], dtype=np.int32)
    begin = np.array([96, 32, 16, 0, 64, 0, 0], dtype=np.int32)     # whole blocks; 16 of 16: no private part
    S = len(lens)
    nb = [-(-int(T) // B) for T in lens]
    N = sum(nb) + 2
    perm = rng.permutation(N).astype(np.int32)
    tables = np.full((S, max(nb)), -1, dtype=np.int32)
    i = 0
    for s, n in enumerate(nb):
        tables[s, :n] = perm[i:i + n]
        i += n
    kp = rng.standard_normal((N, H, B, hd)).astype(np.float16)
    vp = rng.standard_normal((N, H, B, hd)).astype(np.float16)
    q = rng.standard_normal((S, H, hd)).astype(np.float16)
    scale = 1.0 / math.sqrt(hd)
    sl2 = scale * LOG2E
    pcs = np.zeros((S, H, bd.MAX_PREFIX_SPLITS, hd + 4), dtype=np.float32)
    pcs[..., hd] = -np.inf
    for s in range(S):
        for h in range(H):
            for k in range(splits):
                if k == splits // 2 and splits > 1:
                    continue                               # an empty piece: m = -inf, l = 0, o = 0
                l = rng.uniform(0.5, 50.0)
                pcs[s, h, k, hd] = rng.uniform(-4.0, 4.0)
                pcs[s, h, k, hd + 1] = l
                pcs[s, h, k, :hd] = rng.standard_normal(hd) * l
    dev = "cuda"
    pool = pkv.Pool(1, N, B, H, hd, "HND", k_pool=torch.from_numpy(kp).to(dev), v_pool=torch.from_numpy(vp).to(dev))
    out = torch.full((S, H, hd), float("nan"), dtype=torch.float16, device=dev)
    ws = bd.new_workspace(S, H, hd)
    pool.decode_attention_ex(0, torch.from_numpy(q).to(dev), torch.from_numpy(tables).to(dev),
                             torch.from_numpy(lens).to(dev), out, ws, seq_begin=torch.from_numpy(begin).to(dev),
                             pieces=torch.from_numpy(pcs.reshape(-1)).to(dev), splits=splits)
    torch.cuda.synchronize()
    assert bd.workspace_status(ws) == 0
    got = out.cpu().numpy().astype(np.float64)
    ref = np.zeros((S, H, hd))
    for s in range(S):
        T, b0 = int(lens[s]), int(begin[s])
        for h in range(H):
            k = rf.gather_sequence(kp, tables[s], T, h, "HND", H, B, hd)[b0:]
            v = rf.gather_sequence(vp, tables[s], T, h, "HND", H, B, hd)[b0:]
            x = sl2 * (k @ q[s, h].astype(np.float64))
            ms, ls, os_ = [], [], []
            if b0 > 0:
                for kk in range(splits):
                    m = float(pcs[s, h, kk, hd])
                    if m == -np.inf:
                        continue
                    ms.append(m)
                    ls.append(float(pcs[s, h, kk, hd + 1]))
                    os_.append(pcs[s, h, kk, :hd].astype(np.float64))
            M = max(ms + ([x.max()] if len(x) else []))
            num = sum(2.0 ** (m - M) * o for m, o in zip(ms, os_)) + (2.0 ** (x - M)) @ v if len(x) else \
                sum(2.0 ** (m - M) * o for m, o in zip(ms, os_))
            den = sum(2.0 ** (m - M) * l for m, l in zip(ms, ls)) + (np.exp2(x - M).sum() if len(x) else 0.0)
            ref[s, h] = num / den
    assert_close(got, ref, f"merge splits={splits}")


@pytest.mark.parametrize("hd", [64, 256])
def test_pieces_refused_for_other_head_dims(hd):
    """The cascade is built for head_dim 128: other pools refuse pieces before any launch."""
    H, B, S = 2, 16, 2
    kv = torch.zeros((8, H, B, hd), dtype=torch.float16, device="cuda")
    pool = pkv.Pool(1, 8, B, H, hd, "HND", k_pool=kv, v_pool=kv.clone())
    q = torch.zeros((S, H, hd), dtype=torch.float16, device="cuda")
    out = torch.empty_like(q)
    tab = torch.zeros((S, 2), dtype=torch.int32, device="cuda")
    lens = torch.full((S,), 20, dtype=torch.int32, device="cuda")
    begin = torch.full((S,), 16, dtype=torch.int32, device="cuda")
    pcs = torch.zeros((S * H * bd.MAX_PREFIX_SPLITS * (hd + 4),), device="cuda")
    with pytest.raises(bd.PkvError) as e:
        pool.decode_attention_ex(0, q, tab, lens, out, bd.new_workspace(S, H, hd), seq_begin=begin, pieces=pcs,
                                 splits=1)
    assert e.value.code == "UNSUPPORTED", str(e.value)
