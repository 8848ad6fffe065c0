"""Pins of the prefill (chunked causal) attention oracle."""
import numpy as np

from oracle import ref_attn as rf
from tests.test_oracle_attn import _brute, _build_case


def _chunks(lens, C, seed, H=3, D=8, B=4):
    q, kp, vp, tab, ln, ks, vs, B = _build_case(seed, lens, H=H, D=D, B=B, layout="HND")
    rng = np.random.default_rng(seed + 99)
    qc = rng.standard_normal((sum(C), H, D)).astype(np.float16)
    qs = np.concatenate([[0], np.cumsum(C)]).astype(np.int32)
    return qc, qs, kp, vp, tab, ln, ks, vs, B


def test_single_query_chunk_is_decode():
    qc, qs, kp, vp, tab, ln, ks, vs, B = _chunks([9, 14, 5], [1, 1, 1], 1)
    got = rf.prefill_attention(qc, kp, vp, tab, ln, qs, B)
    want = rf.decode_attention(qc, kp, vp, tab, ln, B, layout="HND")
    assert np.allclose(got, want, rtol=1e-13, atol=1e-14)


def test_brute_force_causal():
    lens, C = [9, 14, 5], [4, 14, 2]
    qc, qs, kp, vp, tab, ln, ks, vs, B = _chunks(lens, C, 2)
    got = rf.prefill_attention(qc, kp, vp, tab, ln, qs, B, scale=0.3)
    for s, (T, c) in enumerate(zip(lens, C)):
        for i in range(c):
            p = T - c + i
            row = qs[s] + i
            want = _brute(qc[row:row + 1], [ks[s][:p + 1]], [vs[s][:p + 1]], 0.3)[0]
            assert np.allclose(got[row], want, rtol=1e-12, atol=1e-13)


def test_future_tokens_do_not_matter():
    lens, C = [12], [6]
    qc, qs, kp, vp, tab, ln, ks, vs, B = _chunks(lens, C, 3)
    base = rf.prefill_attention(qc, kp, vp, tab, ln, qs, B)
    # perturb the last cached token: only the last query sees it
    kp2, vp2 = kp.copy(), vp.copy()
    blk, off = tab[0][11 // B], 11 % B
    kp2[blk, :, off] += np.float16(3.0)
    vp2[blk, :, off] -= np.float16(2.0)
    got = rf.prefill_attention(qc, kp2, vp2, tab, ln, qs, B)
    assert np.array_equal(got[:5], base[:5]) and not np.allclose(got[5], base[5])
