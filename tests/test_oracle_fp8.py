"""Pins of the FP8 E4M3 quantisation oracle (oracle/fp8.py)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import fp8
from oracle import ref_attn as rf

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "e4m3.json")))


def test_decode_matches_spec_values():
    for v in GOLD["values"]:
        got = fp8.DECODE[int(v["code"], 16)]
        if v["value"] == "nan":
            assert math.isnan(got)
        else:
            assert got == v["value"], v
    finite = fp8.DECODE[~np.isnan(fp8.DECODE)]
    assert finite.max() == 448.0 and finite.min() == -448.0 and len(finite) == 254


def test_encode_round_trip_all_codes():
    for code in range(256):
        v = fp8.DECODE[code]
        if np.isnan(v):
            continue
        assert fp8.e4m3_encode(np.array([v]))[0] == code


def test_encode_ties_to_even_and_saturation():
    # 1.0625 lies halfway between 1.0 (0x38, even) and 1.125 (0x39): ties go to even
    assert fp8.e4m3_encode(np.array([1.0625]))[0] == 0x38
    assert fp8.e4m3_encode(np.array([1.1875]))[0] == 0x3A     # halfway 1.125 / 1.25 -> 1.25 (even)
    assert fp8.e4m3_encode(np.array([1000.0, -1000.0])).tolist() == [0x7E, 0xFE]
    assert fp8.e4m3_encode(np.array([2.0 ** -10]))[0] == 0x00   # halfway 0 / 2^-9 -> 0 (even)


def test_encode_matches_torch_float8():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    for sc in (1e-3, 1.0, 300.0):
        x = np.clip(rng.standard_normal(100000).astype(np.float32) * sc, -448, 448)
        t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(fp8.e4m3_encode(x), t)


def test_quantize_rows_properties():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((50, 3, 128)).astype(np.float16)
    codes, scales = fp8.quantize_rows(x)
    assert codes.dtype == np.uint8 and scales.dtype == np.float32 and scales.shape == (50, 3)
    # the row maximum maps to +-448 exactly
    assert np.all(np.max(np.abs(fp8.DECODE[codes]), axis=-1) == 448.0)
    deq = fp8.dequantize(codes, scales)
    xf = x.astype(np.float64)
    # relative error of a normal E4M3 value is at most 2^-4 (half of the 3-bit mantissa step)
    big = np.abs(xf) >= scales[..., None].astype(np.float64) * 2.0 ** -6
    assert np.all(np.abs(deq - xf)[big] <= 2.0 ** -4 * np.abs(xf)[big] + 1e-12)
    z, zs = fp8.quantize_rows(np.zeros((2, 128), dtype=np.float16))
    assert np.all(z == 0) and np.all(zs == 1.0)


def test_attention_over_dequantised_values():
    rng = np.random.default_rng(5)
    N, H, B, D = 6, 2, 8, 64
    kc = rng.integers(0, 0x7E, size=(N, H, B, D)).astype(np.uint8)
    vc = rng.integers(0, 0x7E, size=(N, H, B, D)).astype(np.uint8) | (rng.integers(0, 2, size=(N, H, B, D)) << 7).astype(np.uint8)
    ks = rng.uniform(1e-3, 1e-2, size=(N, H, B)).astype(np.float32)
    vs = rng.uniform(1e-3, 1e-2, size=(N, H, B)).astype(np.float32)
    q = rng.standard_normal((2, H, D)).astype(np.float16)
    tables = np.array([[3, 1, 4], [0, 5, 2]], dtype=np.int32)
    lens = np.array([19, 9], dtype=np.int32)
    got = fp8.decode_attention(q, kc, vc, ks, vs, tables, lens, B)
    kd = fp8.dequantize(kc, ks)
    vd = fp8.dequantize(vc, vs)
    want = rf.decode_attention(q, kd, vd, tables, lens, B, layout="HND")
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14)


def test_append_and_copy_quantised():
    rng = np.random.default_rng(6)
    N, H, B, D = 4, 2, 8, 64
    kc = np.zeros((1, N, H, B, D), dtype=np.uint8)
    vc = kc.copy()
    ks = np.zeros((1, N, H, B), dtype=np.float32)
    vs = ks.copy()
    kn = rng.standard_normal((2, H, D)).astype(np.float16)
    vn = rng.standard_normal((2, H, D)).astype(np.float16)
    fp8.append_kv(kc[0], vc[0], ks[0], vs[0], kn, vn, [9, -1], B)
    q, s = fp8.quantize_rows(kn[0])
    assert np.array_equal(kc[0, 1, :, 1], q) and np.array_equal(ks[0, 1, :, 1], s)
    assert np.count_nonzero(kc) == np.count_nonzero(q)
    fp8.copy_blocks(kc, vc, ks, vs, [(1, 3)])
    assert np.array_equal(kc[:, 3], kc[:, 1]) and np.array_equal(vs[:, 3], vs[:, 1])


def test_nhd_layout_is_the_hnd_one_transposed():
    """The two code layouts hold the same rows: an NHD pool that is the HND pool with its
    head and in-block axes swapped gives the same attention bit for bit, and an append
    writes the same codes (at the swapped place) and the same scales. The NHD indexing is
    the one that gathers by hand below, too."""
    rng = np.random.default_rng(8)
    N, H, B, D = 7, 3, 8, 64
    kc = rng.integers(0, 0x7E, size=(N, H, B, D)).astype(np.uint8) | (rng.integers(0, 2, size=(N, H, B, D)) << 7).astype(np.uint8)
    vc = rng.integers(0, 0x7E, size=(N, H, B, D)).astype(np.uint8) | (rng.integers(0, 2, size=(N, H, B, D)) << 7).astype(np.uint8)
    ks = rng.uniform(1e-3, 1e-2, size=(N, H, B)).astype(np.float32)
    vs = rng.uniform(1e-3, 1e-2, size=(N, H, B)).astype(np.float32)
    q = rng.standard_normal((3, H, D)).astype(np.float16)
    tables = np.array([[3, 1, 4], [0, 5, 2], [6, 0, 0]], dtype=np.int32)
    lens = np.array([19, 17, 5], dtype=np.int32)
    kn_, vn_ = np.ascontiguousarray(kc.transpose(0, 2, 1, 3)), np.ascontiguousarray(vc.transpose(0, 2, 1, 3))
    hnd = fp8.decode_attention(q, kc, vc, ks, vs, tables, lens, B)
    nhd = fp8.decode_attention(q, kn_, vn_, ks, vs, tables, lens, B, layout="NHD")
    assert np.array_equal(hnd, nhd)
    # by hand: sequence 1, head 2 gathers rows (block, offset) through the NHD codes
    rows = [(int(tables[1][t // B]), t % B) for t in range(int(lens[1]))]
    k = np.stack([fp8.DECODE[kn_[b, o, 2]] * float(ks[b, 2, o]) for b, o in rows])
    v = np.stack([fp8.DECODE[vn_[b, o, 2]] * float(vs[b, 2, o]) for b, o in rows])
    assert np.allclose(nhd[1, 2], rf.attend(q[1, 2], k, v, 1.0 / np.sqrt(D)), rtol=1e-12, atol=1e-14)
    # an append: the same codes at the swapped place, the same scales
    kn = rng.standard_normal((2, H, D)).astype(np.float16)
    vn = rng.standard_normal((2, H, D)).astype(np.float16)
    a = [x.copy() for x in (kc, vc, ks, vs)]
    b = [kn_.copy(), vn_.copy(), ks.copy(), vs.copy()]
    fp8.append_kv(*a, kn, vn, [13, 50], B)
    fp8.append_kv(*b, kn, vn, [13, 50], B, layout="NHD")
    assert np.array_equal(a[0].transpose(0, 2, 1, 3), b[0]) and np.array_equal(a[1].transpose(0, 2, 1, 3), b[1])
    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
    assert not np.array_equal(a[0], kc)


# --------------------------------------------------------------------------- planted mistakes
# The pins above, as checks of a given encoder / quantiser, and copies of the oracle's
# quantiser with one plausible slip each: every slip makes at least one check fail.

def _check_round_trip(encode):
    codes = [c for c in range(256) if not np.isnan(fp8.DECODE[c])]
    return all(int(encode(np.array([fp8.DECODE[c]]))[0]) == c for c in codes)


def _check_ties_and_saturation(encode):
    return (int(encode(np.array([1.0625]))[0]) == 0x38 and int(encode(np.array([1.1875]))[0]) == 0x3A
            and encode(np.array([1000.0, -1000.0])).tolist() == [0x7E, 0xFE]
            and int(encode(np.array([2.0 ** -10]))[0]) == 0x00)


def _check_torch(encode):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    for sc in (1e-3, 1.0, 300.0):
        x = np.clip(rng.standard_normal(20000).astype(np.float32) * sc, -448, 448)
        t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        if not np.array_equal(encode(x), t):
            return False
    return True


def _check_rows(quantize):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((50, 3, 128)).astype(np.float16)
    codes, scales = quantize(x)
    if scales.shape != (50, 3) or not np.all(np.max(np.abs(fp8.DECODE[codes]), axis=-1) == 448.0):
        return False
    deq = fp8.dequantize(codes, scales)
    xf = x.astype(np.float64)
    big = np.abs(xf) >= scales[..., None].astype(np.float64) * 2.0 ** -6
    return bool(np.all(np.abs(deq - xf)[big] <= 2.0 ** -4 * np.abs(xf)[big] + 1e-12))


def _mutant_encode(kind):
    vals = fp8.DECODE[:0x7F]

    def encode(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x) if kind == "no_saturation" else np.minimum(np.abs(x), 448.0)
        lo = np.clip(np.searchsorted(vals, a, side="right") - 1, 0, 0x7E)
        hi = np.minimum(lo + 1, 0x7E)
        below, above = a - vals[lo], vals[hi] - a
        if kind == "ties_away":
            pick_hi = (above < below) | ((above == below) & (hi != lo))
        elif kind == "truncate":
            pick_hi = np.zeros(a.shape, dtype=bool)
        else:
            pick_hi = (above < below) | ((above == below) & (hi != lo) & ((hi & 1) == 0))
        code = np.where(pick_hi, hi, lo).astype(np.int64)
        if kind == "no_saturation":
            code = np.where(a > 448.0, 0x7F, code)
        sign = np.signbit(x).astype(np.int64) << 7
        if kind == "sign_lost_at_zero":
            sign = np.where(code == 0, 0, sign)
        return (code | sign).astype(np.uint8)
    return encode


def _mutant_quantize(kind):
    def quantize(x16):
        x = np.asarray(x16, dtype=np.float16).astype(np.float32)
        if kind == "amax_over_heads":
            amax = np.broadcast_to(np.max(np.abs(x), axis=(-2, -1))[..., None], x.shape[:-1])
        else:
            amax = np.max(np.abs(x), axis=-1)
        div = np.float32(256.0) if kind == "scale_256" else np.float32(448.0)
        scale = np.where(amax > 0, amax / div, np.float32(1.0)).astype(np.float32)
        y = (x / scale[..., None]).astype(np.float32)
        return fp8.e4m3_encode(y), scale
    return quantize


@pytest.mark.parametrize("kind", ["ties_away", "truncate", "no_saturation", "sign_lost_at_zero"])
def test_planted_encoder_mistake_is_caught(kind):
    enc = _mutant_encode(kind)
    assert not (_check_round_trip(enc) and _check_ties_and_saturation(enc) and _check_torch(enc)), kind


@pytest.mark.parametrize("kind", ["scale_256", "amax_over_heads"])
def test_planted_quantiser_mistake_is_caught(kind):
    assert not _check_rows(_mutant_quantize(kind)), kind


def test_unmutated_quantiser_copies_pass():
    enc = _mutant_encode("none")
    assert _check_round_trip(enc) and _check_ties_and_saturation(enc) and _check_torch(enc)
    assert _check_rows(_mutant_quantize("none"))
