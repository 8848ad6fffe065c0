"""GPU parity of the shared-prefix (cascade) decode on an FP8 E4M3 cache.

The E4M3 prefix pass (pkv_prefix_attention on an E4M3 pool) is checked piece by
piece against float64 on the dequantised keys and values (code x row scale): o / l
is the softmax-weighted mean of V over the piece's keys and m + log2(l) is
log2 sum_t 2^(scale log2(e) q.K_t). The whole cascade (prefix pass, then the
private pass of pkv_decode_attention_ex) is checked against the float64 E4M3
oracle's attention, with NaN codes and scales past every context.
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
from oracle import fp8  # noqa: E402
from oracle import ref_attn as rf  # noqa: E402
from tests.test_gpu_cascade import forked_spec  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2
D = 128
LOG2E = 1.4426950408889634


def assert_close(got, ref, what):
    err = np.abs(got.astype(np.float64) - ref)
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {np.nanmax(err):.3e}"


class Q8Case:
    """E4M3 codes (no NaN code inside a context) and row scales U[0.001, 0.01]; codes 0x7F
    and NaN scales past each context. Tables as the fp16 cascade tests build them."""

    def __init__(self, spec, H=4, B=16, seed=0):
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
        perm = rng.permutation(N).astype(np.int32)
        self.tables = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
        self.lens = np.array([T for _, _, T in spec], dtype=np.int32)
        kc = rng.integers(0, 256, size=(N, H, B, D), dtype=np.uint8)
        vc = rng.integers(0, 256, size=(N, H, B, D), dtype=np.uint8)
        for c_ in (kc, vc):
            c_[(c_ & 0x7F) == 0x7F] ^= 1
        ks = rng.uniform(0.001, 0.01, size=(N, H, B)).astype(np.float32)
        vs = rng.uniform(0.001, 0.01, size=(N, H, B)).astype(np.float32)
        for s, T in enumerate(self.lens):
            nb = -(-int(T) // B)
            off = int(T) - (nb - 1) * B
            if off < B:
                b = self.tables[s, nb - 1]
                kc[b, :, off:] = 0x7F
                vc[b, :, off:] = 0xFF
                ks[b, :, off:] = np.nan
                vs[b, :, off:] = np.nan
        self.kc, self.vc, self.ks, self.vs = kc, vc, ks, vs
        self.q = rng.standard_normal((S, H, D)).astype(np.float16)
        self.H, self.B, self.S, self.N = H, B, S, N
        self.scale = 1.0 / math.sqrt(D)
        dev = "cuda"
        self.pool = pkv.Pool(1, N, B, H, D, "HND", k_pool=torch.from_numpy(kc).to(dev),
                             v_pool=torch.from_numpy(vc).to(dev), kv_dtype="e4m3",
                             k_scale=torch.from_numpy(ks).to(dev), v_scale=torch.from_numpy(vs).to(dev))
        self.qd = torch.from_numpy(self.q).to(dev)
        self.tab_d = torch.from_numpy(self.tables).to(dev)
        self.lens_d = torch.from_numpy(self.lens).to(dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pieces = torch.full((bd.prefix_pieces_bytes(S, H, D) // 4,), float("nan"), device=dev)
        self.ws = bd.new_workspace(S, H, D)

    def plan(self):
        g, b = bd.cascade_plan(self.tables, self.lens, self.B)
        return g.copy(), b.copy()

    def prefix(self, groups, splits):
        gd = torch.from_numpy(np.ascontiguousarray(groups, dtype=np.int32)).cuda()
        self.pool.prefix_attention(0, self.qd, gd, len(groups), splits, self.tab_d, self.pieces, self.status)

    def decode(self, begin, splits):
        out = torch.full_like(self.qd, float("nan"))
        bdv = torch.from_numpy(np.ascontiguousarray(begin, dtype=np.int32)).cuda() if begin is not None else None
        self.pool.decode_attention_ex(0, self.qd, self.tab_d, self.lens_d, out, self.ws, seq_begin=bdv,
                                      pieces=self.pieces if begin is not None else None, splits=splits)
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def oracle(self):
        return fp8.decode_attention(self.q, self.kc, self.vc, self.ks, self.vs, self.tables, self.lens, self.B)

    def keys(self, s, h, t0, t1):
        """Dequantised K and V rows of sequence s, head h, tokens [t0, t1) (float64)."""
        blk = [int(self.tables[s][t // self.B]) for t in range(t0, t1)]
        off = [t % self.B for t in range(t0, t1)]
        k = fp8.dequantize(self.kc[blk, h, off], self.ks[blk, h, off])
        v = fp8.dequantize(self.vc[blk, h, off], self.vs[blk, h, off])
        return k, v


@pytest.mark.parametrize("splits", [1, 3])
def test_e4m3_prefix_pieces(splits):
    """Every piece against its keys: a 1040-token prefix (a ragged last 64-key tile), a
    second group of 70 members (two CTAs per split), and splits with no keys."""
    rng = np.random.default_rng(5)
    B = 16
    spec = forked_spec(5, 65, 40, B, rng) + [(None, 0, 300)] + forked_spec(70, 4, 100, B, rng)
    spec[6:] = [(6, 4, T) if src is not None else (None, 0, T) for src, _, T in spec[6:]]
    c = Q8Case(spec, H=2, B=B, seed=6)
    groups, begin = c.plan()
    assert groups[:, :3].tolist() == [[0, 5, 1040], [6, 70, 64]]
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
                    assert_close(o / l, rf.attend(c.q[s, h], kk, vv, c.scale), f"piece {(s, h, k)}")


@pytest.mark.parametrize("B", [8, 16, 64, 256, 512])
def test_e4m3_cascade_matches_oracle(B):
    """Two groups, unshared sequences, and a member whose whole context is the prefix."""
    rng = np.random.default_rng(B + 100)
    nsh = max(1, 600 // B)
    spec = forked_spec(6, nsh, 3 * B, B, rng)
    spec += [(None, 0, int(rng.integers(1, 700))), (None, 0, 5)]
    g2 = len(spec)
    spec += [(None, 0, 2 * B + 7), (g2, 2, 2 * B + 3), (g2, 2, 2 * B)]     # the last: no private tokens
    c = Q8Case(spec, H=4, B=B, seed=B + 3)
    groups, begin = c.plan()
    assert len(groups) == 2 and begin[-1] == c.lens[-1]
    splits = bd.prefix_splits(len(groups), c.H, int(groups[:, 2].max()))
    c.prefix(groups, splits)
    got = c.decode(begin, splits)
    assert int(c.status.item()) == 0 and bd.workspace_status(c.ws) == 0
    ref = c.oracle()
    assert_close(got, ref, f"E4M3 cascade B={B}")
    assert_close(c.decode(None, 0), ref, f"E4M3 plain B={B}")


def test_e4m3_prefix_pass_early_start_identical():
    """Started early behind a preceding attention launch, the E4M3 prefix pass writes the same
    pieces, bit for bit, as started after it."""
    rng = np.random.default_rng(9)
    B = 16
    spec = forked_spec(8, 40, 60, B, rng)
    c = Q8Case(spec, H=4, B=B, seed=10)
    groups, _ = c.plan()
    c.prefix(groups, 2)
    torch.cuda.synchronize()
    ref = c.pieces.clone()
    gd = torch.from_numpy(np.ascontiguousarray(groups, dtype=np.int32)).cuda()
    c.pieces.fill_(float("nan"))
    c.pool.decode_attention_ex(0, c.qd, c.tab_d, c.lens_d, torch.empty_like(c.qd), c.ws)
    c.pool.prefix_attention(0, c.qd, gd, len(groups), 2, c.tab_d, c.pieces, c.status, flags=bd.ATTN_INPUTS_EARLY)
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    f, n = int(groups[0, 0]), int(groups[0, 1])
    got = c.pieces.view(c.S, c.H, bd.MAX_PREFIX_SPLITS, D + 4)[f:f + n, :, :2]
    want = ref.view(c.S, c.H, bd.MAX_PREFIX_SPLITS, D + 4)[f:f + n, :, :2]
    assert torch.equal(got, want)
