"""Pins of the prefill (chunked causal) attention oracle."""
import numpy as np
import pytest

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


# --------------------------------------------------------------------------- planted mistakes
# The pins above as checks of a given prefill function, and copies of the oracle with one
# plausible slip each: every slip makes at least one check fail.

def _check_decode(prefill):
    qc, qs, kp, vp, tab, ln, ks, vs, B = _chunks([9, 14, 5], [1, 1, 1], 1)
    want = rf.decode_attention(qc, kp, vp, tab, ln, B, layout="HND")
    return np.allclose(prefill(qc, kp, vp, tab, ln, qs, B), want, rtol=1e-13, atol=1e-14)


def _check_brute(prefill):
    lens, C = [9, 14, 5], [4, 14, 2]
    qc, qs, kp, vp, tab, ln, ks, vs, B = _chunks(lens, C, 2)
    got = prefill(qc, kp, vp, tab, ln, qs, B, scale=0.3)
    for s, (T, c) in enumerate(zip(lens, C)):
        for i in range(c):
            p, row = T - c + i, qs[s] + i
            want = _brute(qc[row:row + 1], [ks[s][:p + 1]], [vs[s][:p + 1]], 0.3)[0]
            if not np.allclose(got[row], want, rtol=1e-12, atol=1e-13):
                return False
    return True


def _check_future(prefill):
    qc, qs, kp, vp, tab, ln, ks, vs, B = _chunks([12], [6], 3)
    base = prefill(qc, kp, vp, tab, ln, qs, B)
    kp2, vp2 = kp.copy(), vp.copy()
    blk, off = tab[0][11 // B], 11 % B
    kp2[blk, :, off] += np.float16(3.0)
    vp2[blk, :, off] -= np.float16(2.0)
    got = prefill(qc, kp2, vp2, tab, ln, qs, B)
    return bool(np.array_equal(got[:5], base[:5]) and not np.allclose(got[5], base[5]))


def _mutant(kind):
    def prefill(q, kp, vp, tables, lens, q_start, B, layout="HND", scale=None):
        R, H, D = q.shape
        scale = rf.default_scale(D) if scale is None else scale
        out = np.zeros((R, H, D))
        for s in range(len(lens)):
            r0, r1 = int(q_start[s]), int(q_start[s + 1])
            C, T = r1 - r0, int(lens[s])
            if C == 0:
                continue
            pos = np.arange(0, C) if kind == "positions_from_zero" else np.arange(T - C, T)
            rows = np.clip(np.arange(r0, r1) + (1 if kind == "rows_shifted" else 0), 0, R - 1)
            for h in range(H):
                k = rf.gather_sequence(kp, tables[s], T, h, layout, H, B, D)
                v = rf.gather_sequence(vp, tables[s], T, h, layout, H, B, D)
                x = scale * (q[rows, h].astype(np.float64) @ k.T)
                if kind == "mask_off_by_one":
                    x[np.arange(T)[None, :] >= pos[:, None]] = -np.inf
                elif kind != "no_mask":
                    x[np.arange(T)[None, :] > pos[:, None]] = -np.inf
                x = x - x.max(axis=1, keepdims=True)
                w = np.exp(x)
                w /= w.sum(axis=1, keepdims=True)
                out[r0:r1, h] = w @ v
        return out
    return prefill



@pytest.mark.parametrize("kind", ["mask_off_by_one", "positions_from_zero", "no_mask", "rows_shifted"])
def test_planted_prefill_mistake_is_caught(kind):
    m = _mutant(kind)
    results = []
    for check in (_check_decode, _check_brute, _check_future):
        with np.errstate(invalid="ignore", divide="ignore"):
            try:
                results.append(check(m))
            except Exception:
                results.append(False)
    assert not all(results), kind


def test_unmutated_prefill_copy_passes():
    m = _mutant("none")
    assert _check_decode(m) and _check_brute(m) and _check_future(m)
