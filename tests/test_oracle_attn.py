"""Pins of the attention / append / copy oracle (oracle/ref_attn.py, oracle/ref_attn.c).

What pins it to something other than itself:

* special cases with a known answer (T = 1, equal keys, scale 0, q = 0, one
  dominant key, a two-token case with exact weights 3/4 and 1/4);
* brute force on tiny inputs: pure-Python loops over a CONTIGUOUS copy of each
  sequence that the test scatters into the pool with its own placement;
* invariants: physical-block relabelling, block layout, block size,
  shared prefix = private copy, weights summing to 1;
* two independent implementations (NumPy and C) agreeing to 1e-12, and the C
  binary16 decoder matching NumPy's on all 65,536 bit patterns;
* a planted-mistake check: each plausible slip, planted in a copy of the
  oracle, makes at least one of these checks fail.
"""
import math

import numpy as np
import pytest

from oracle import ref_attn as rf
from oracle import ref_attn_c as rc


def _build_case(seed, lens, H=3, D=8, B=4, extra_blocks=3, layout="NHD"):
    """Contiguous per-sequence K/V, scattered into a shuffled pool by the test itself.

    The token data depends only on (seed, lens, H, D), so the same tokens can be
    laid out with another block size or layout.
    """
    rng = np.random.default_rng(seed)
    S = len(lens)
    q = rng.standard_normal((S, H, D)).astype(np.float16)
    kseq = [rng.standard_normal((t, H, D)).astype(np.float16) for t in lens]
    vseq = [rng.standard_normal((t, H, D)).astype(np.float16) for t in lens]
    rng2 = np.random.default_rng([seed, B])
    nb = [-(-t // B) for t in lens]
    N = sum(nb) + extra_blocks
    perm = rng2.permutation(N)
    maxb = max(nb + [1])
    tables = -np.ones((S, maxb), dtype=np.int32)
    kpool = rng2.standard_normal((N, B, H, D)).astype(np.float16)   # garbage everywhere else
    vpool = rng2.standard_normal((N, B, H, D)).astype(np.float16)
    i = 0
    for s, t in enumerate(lens):
        for j in range(nb[s]):
            tables[s, j] = perm[i]
            i += 1
        for tok in range(t):
            blk = tables[s, tok // B]
            kpool[blk, tok % B] = kseq[s][tok]
            vpool[blk, tok % B] = vseq[s][tok]
    if layout == "HND":
        kpool = np.ascontiguousarray(kpool.transpose(0, 2, 1, 3))
        vpool = np.ascontiguousarray(vpool.transpose(0, 2, 1, 3))
    return q, kpool, vpool, tables, np.asarray(lens, dtype=np.int32), kseq, vseq, B


def _brute(q, kseq, vseq, scale):
    """Pure-Python loops, exp without max subtraction (values here are small)."""
    S, H, D = q.shape
    out = np.zeros((S, H, D))
    for s in range(S):
        T = kseq[s].shape[0]
        for h in range(H):
            if T == 0:
                continue
            w = []
            for t in range(T):
                dot = 0.0
                for d in range(D):
                    dot += float(q[s, h, d]) * float(kseq[s][t, h, d])
                w.append(math.exp(scale * dot))
            z = sum(w)
            for d in range(D):
                out[s, h, d] = sum(w[t] * float(vseq[s][t, h, d]) for t in range(T)) / z
    return out


# --------------------------------------------------------------------------- checks
# Each returns True when the oracle passes; the planted-mistake test reuses them.

def check_brute_force(mod=rf):
    ok = True
    for layout in ("NHD", "HND"):
        q, kp, vp, tab, lens, ks, vs, B = _build_case(1, [1, 3, 4, 5, 9, 0], layout=layout)
        scale = 0.37
        got = mod.decode_attention(q, kp, vp, tab, lens, B, layout=layout, scale=scale)
        ok &= np.allclose(got, _brute(q, ks, vs, scale), rtol=1e-12, atol=1e-13)
        # default scale: 1/sqrt(head_dim), the reading for the scale the pages leave open
        got = mod.decode_attention(q, kp, vp, tab, lens, B, layout=layout)
        ok &= np.allclose(got, _brute(q, ks, vs, 8 ** -0.5), rtol=1e-12, atol=1e-13)
    return bool(ok)


def check_special_cases(mod=rf):
    ok = True
    q, kp, vp, tab, lens, ks, vs, B = _build_case(2, [1, 7])
    out = mod.decode_attention(q, kp, vp, tab, lens, B)
    ok &= np.array_equal(out[0], vs[0][0].astype(np.float64))   # T = 1: exactly V[0]
    out0 = mod.decode_attention(q, kp, vp, tab, lens, B, scale=0.0)          # scale 0: mean of V
    ok &= np.allclose(out0[1], vs[1].astype(np.float64).mean(axis=0), rtol=1e-12, atol=1e-14)
    qz = np.zeros_like(q)
    outz = mod.decode_attention(qz, kp, vp, tab, lens, B)                    # q = 0: mean of V
    ok &= np.allclose(outz[1], vs[1].astype(np.float64).mean(axis=0), rtol=1e-12, atol=1e-14)
    # all keys equal: mean of V
    kp2 = kp.copy()
    for t in range(7):
        kp2[tab[1, t // B], t % B] = ks[1][0]
    oute = mod.decode_attention(q, kp2, vp, tab, lens, B)
    ok &= np.allclose(oute[1], vs[1].astype(np.float64).mean(axis=0), rtol=1e-12, atol=1e-14)
    # one key with a huge dot product: that token's V
    kp3 = kp.copy()
    t_hot = 5
    kp3[tab[1, t_hot // B], t_hot % B] = (q[1] * np.float16(60)).astype(np.float16)
    outh = mod.decode_attention(q, kp3, vp, tab, lens, B)
    ok &= np.allclose(outh[1], vs[1][t_hot].astype(np.float64), rtol=1e-9, atol=1e-9)
    return bool(ok)


def check_two_token_closed_form(mod=rf):
    """x0 = ln 3, x1 = 0 gives weights exactly 3/4 and 1/4."""
    H, D, B = 2, 4, 4
    kp = np.zeros((2, B, H, D), dtype=np.float16)
    vp = np.zeros((2, B, H, D), dtype=np.float16)
    q = np.zeros((1, H, D), dtype=np.float16)
    q[0, 1, 2] = 2.0
    kp[1, 0, 1, 2] = 1.0                 # token 0 lives in physical block 1
    vp[1, 0, 1] = [1.0, -2.0, 0.5, 4.0]
    vp[1, 1, 1] = [3.0, 2.0, -1.5, 0.0]
    tab = np.array([[1, 0]], dtype=np.int32)
    out = mod.decode_attention(q, kp, vp, tab, np.array([2], dtype=np.int32), B, scale=math.log(3.0) / 2)
    want = 0.75 * np.array([1.0, -2.0, 0.5, 4.0]) + 0.25 * np.array([3.0, 2.0, -1.5, 0.0])
    return bool(np.allclose(out[0, 1], want, rtol=1e-14, atol=1e-14))


def check_invariants(mod=rf):
    ok = True
    q, kp, vp, tab, lens, ks, vs, B = _build_case(3, [6, 13, 2, 9])
    base = mod.decode_attention(q, kp, vp, tab, lens, B)
    # relabel physical blocks: data moves with its id
    N = kp.shape[0]
    pi = np.random.default_rng(9).permutation(N)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[pi] = kp
    vp2[pi] = vp
    tab2 = np.where(tab >= 0, pi[np.maximum(tab, 0)], -1).astype(np.int32)
    ok &= np.array_equal(mod.decode_attention(q, kp2, vp2, tab2, lens, B), base)
    # layout
    q3, kp3, vp3, tab3, _, _, _, _ = _build_case(3, [6, 13, 2, 9], layout="HND")
    ok &= np.array_equal(mod.decode_attention(q3, kp3, vp3, tab3, lens, B, layout="HND"), base)
    # block size: same token data at B = 2 and B = 8
    for B2 in (2, 8):
        qq, kk, vv, tt, _, _, _, _ = _build_case(3, [6, 13, 2, 9], B=B2)
        ok &= np.array_equal(mod.decode_attention(qq, kk, vv, tt, lens, B2), base)
    # shared prefix = private copy: seq 1 read through copies of its first two blocks
    used = set(int(b) for b in tab[tab >= 0])
    spare = [b for b in range(N) if b not in used]
    kp4, vp4 = kp.copy(), vp.copy()
    tab_priv = tab[1].copy()
    for j in range(2):
        kp4[spare[j]] = kp[tab[1, j]]
        vp4[spare[j]] = vp[tab[1, j]]
        tab_priv[j] = spare[j]
    priv = mod.decode_attention(q[1:2], kp4, vp4, tab_priv[None], lens[1:2], B)
    ok &= np.array_equal(priv[0], base[1])
    # two sequences sharing all blocks give the same output
    lens_s = np.array([9, 9], dtype=np.int32)
    tab_s = np.stack([tab[1, :3], tab[1, :3]]).astype(np.int32)
    shared = mod.decode_attention(np.stack([q[1], q[1]]), kp, vp, tab_s, lens_s, B)
    ok &= np.array_equal(shared[0], shared[1])
    # weights sum to one
    for s in range(len(lens)):
        for h in range(q.shape[1]):
            k = mod.gather_sequence(kp, tab[s], int(lens[s]), h, "NHD", q.shape[1], B, q.shape[2])
            if k.shape[0]:
                w = mod.softmax_weights(q[s, h], k, 0.5)
                ok &= abs(w.sum() - 1.0) < 1e-12 and (w >= 0).all()
    return bool(ok)


# --------------------------------------------------------------------------- tests

def test_brute_force():
    assert check_brute_force()


def test_special_cases():
    assert check_special_cases()


def test_two_token_closed_form():
    assert check_two_token_closed_form()


def test_invariants():
    assert check_invariants()


def test_empty_context_gives_zero():
    q, kp, vp, tab, lens, ks, vs, B = _build_case(4, [0, 3])
    out = rf.decode_attention(q, kp, vp, tab, lens, B)
    assert np.all(out[0] == 0.0)


def test_c_half_decoder_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([rc.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[np.isinf(want)], want[np.isinf(want)])


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_c_oracle_matches_numpy_oracle(layout):
    q, kp, vp, tab, lens, ks, vs, B = _build_case(5, [1, 17, 40, 0, 33, 8], H=4, D=64, B=16, layout=layout)
    a = rf.decode_attention(q, kp, vp, tab, lens, B, layout=layout)
    b = rc.decode_attention(q, kp, vp, tab, lens, B, layout=layout)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)
    pairs = [(1, 2), (4, 0)]
    c = rc.decode_attention(q, kp, vp, tab, lens, B, layout=layout, pairs=pairs)
    for s, h in pairs:
        assert np.allclose(c[s, h], a[s, h], rtol=1e-12, atol=1e-13)


def test_c_oracle_rejects_bad_block():
    q, kp, vp, tab, lens, ks, vs, B = _build_case(6, [5])
    tab[0, 1] = kp.shape[0]
    with pytest.raises(ValueError):
        rc.decode_attention(q, kp, vp, tab, lens, B)


def test_append_oracle_bit_exact_with_canary():
    H, D, B, N = 3, 8, 4, 5
    for layout in ("NHD", "HND"):
        shape = (N, B, H, D) if layout == "NHD" else (N, H, B, D)
        kp = np.full(shape, np.uint16(0xFFFF), dtype=np.uint16).view(np.float16)
        vp = kp.copy()
        rng = np.random.default_rng(7)
        kn = rng.standard_normal((4, H, D)).astype(np.float16)
        vn = rng.standard_normal((4, H, D)).astype(np.float16)
        slots = [7, -1, 0, 19]
        rf.append_kv(kp, vp, kn, vn, slots, B, layout)
        kb = kp.view(np.uint16)
        for i, slot in enumerate(slots):
            if slot < 0:
                continue
            blk, off = divmod(slot, B)
            got = kb[blk, off] if layout == "NHD" else kb[blk, :, off]
            assert np.array_equal(got, kn[i].view(np.uint16))
        written = sum(1 for s in slots if s >= 0) * H * D
        assert np.count_nonzero(kb != 0xFFFF) <= written
        assert np.count_nonzero(kb == 0xFFFF) >= kb.size - written


def test_copy_blocks_oracle():
    rng = np.random.default_rng(8)
    kp = rng.standard_normal((3, 6, 4, 2, 8)).astype(np.float16)
    vp = rng.standard_normal((3, 6, 4, 2, 8)).astype(np.float16)
    k0, v0 = kp.copy(), vp.copy()
    rf.copy_blocks(kp, vp, [(1, 4), (1, 5), (0, 2)])
    for src, dst in [(1, 4), (1, 5), (0, 2)]:
        assert np.array_equal(kp[:, dst].view(np.uint16), k0[:, src].view(np.uint16))
        assert np.array_equal(vp[:, dst].view(np.uint16), v0[:, src].view(np.uint16))
    for b in (0, 1, 3):
        assert np.array_equal(kp[:, b], k0[:, b]) and np.array_equal(vp[:, b], v0[:, b])


# --------------------------------------------------------------------------- planted mistakes

class _Mutant:
    """A copy of the oracle's public functions with one planted slip."""

    def __init__(self, kind):
        self.kind = kind

    def kv_row(self, layout, block, slot, head, H, B):
        if self.kind == "slot_head_swapped":
            return (block * B + head) * H + slot if layout == "NHD" else rf.kv_row(layout, block, slot, head, H, B)
        if self.kind == "block_index_off_by_one":
            return rf.kv_row(layout, block + 1 if block + 1 < 10 else block, slot, head, H, B)
        return rf.kv_row(layout, block, slot, head, H, B)

    def gather_sequence(self, pool, row, T, h, layout, H, B, D):
        rows = rf.layer_rows(pool, D)
        if self.kind == "token_divmod_swapped":
            idx = [self.kv_row(layout, int(row[t % B] if t % B < len(row) else row[0]), t // B, h, H, B)
                   for t in range(T)]
        else:
            idx = [self.kv_row(layout, int(row[t // B]), t % B, h, H, B) for t in range(T)]
        idx = [min(max(i, 0), rows.shape[0] - 1) for i in idx]
        return rows[np.asarray(idx, dtype=np.int64)].astype(np.float64)

    def softmax_weights(self, q, k, scale):
        x = scale * (k @ q.astype(np.float64))
        if self.kind == "sign_flipped":
            x = -x
        x = x - x.max()
        w = np.exp(x)
        if self.kind == "not_normalised":
            return w
        return w / w.sum()

    def decode_attention(self, q, kp, vp, tab, lens, B, layout="NHD", scale=None, pairs=None):
        S, H, D = q.shape
        if scale is None:
            scale = 1.0 / D if self.kind == "scale_1_over_d" else 1.0 / math.sqrt(D)
        out = np.zeros((S, H, D))
        for s in range(S):
            for h in range(H):
                T = int(lens[s])
                if self.kind == "last_token_dropped":
                    T = max(T - 1, 0) if T > 1 else T
                if T == 0:
                    continue
                k = self.gather_sequence(kp, tab[s], T, h, layout, H, B, D)
                v = self.gather_sequence(vp, tab[s], T, h, layout, H, B, D)
                if self.kind == "k_v_swapped":
                    k, v = v, k
                out[s, h] = self.softmax_weights(q[s, h], k, scale) @ v
        return out


@pytest.mark.parametrize("kind", ["slot_head_swapped", "block_index_off_by_one", "token_divmod_swapped",
                                  "sign_flipped", "not_normalised", "scale_1_over_d", "last_token_dropped",
                                  "k_v_swapped"])
def test_planted_mistake_is_caught(kind):
    m = _Mutant(kind)
    checks = [check_brute_force, check_special_cases, check_two_token_closed_form, check_invariants]
    results = []
    for c in checks:
        try:
            results.append(c(m))
        except Exception:
            results.append(False)
    assert not all(results), f"planted mistake {kind} not caught"


def test_unmutated_copy_passes():
    m = _Mutant("none")
    for c in (check_brute_force, check_special_cases, check_two_token_closed_form, check_invariants):
        assert c(m)
