"""FP8 E4M3 KV quantisation oracle (test infrastructure only).

Quantised KV halves the bytes per token (m.lqnn.cn/news/240480 §6.2: 8,192 bytes
per token per layer instead of 16,384; hnwysp.cn/news/103996 §5.4; icman.com.cn/news/78786
§1.3). The pages name INT8/INT4 storage but no format; the reading taken here:

* codes are FP8 E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
  no infinities, largest finite 448, S.1111.111 = NaN), decoded exactly;
* one fp32 scale per (token, head) row: scale = amax(|row|) / 448 in fp32
  (1 when the row is all zeros), code = round-to-nearest-even of (x / scale)
  computed in fp32, saturated to +-448 -- the same operations, in the same
  precision, as the kernel that writes the cache;
* the attention over a quantised cache is the plain definition applied to the
  dequantised values code * scale (exact in float64).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode_table() -> np.ndarray:
    """float64 value of every byte 0..255 read as E4M3 (NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            vals[code] = np.nan
        elif exp == 0:
            vals[code] = sign * man * 2.0 ** -9            # subnormal: man/8 * 2^(1-7)
        else:
            vals[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return vals


DECODE = e4m3_decode_table()
# finite non-negative codes sorted by value (0x00..0x7E are increasing)
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALS = DECODE[:0x7F]


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even to E4M3 with saturation to +-448 (x finite, float32 or float64)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    # index of the largest representable value <= a
    lo = np.clip(np.searchsorted(_POS_VALS, a, side="right") - 1, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    vlo, vhi = _POS_VALS[lo], _POS_VALS[hi]
    below = a - vlo
    above = vhi - a
    pick_hi = (above < below) | ((above == below) & (hi != lo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    sign = np.signbit(x).astype(np.int64) << 7        # the sign survives rounding to zero
    return (code | sign).astype(np.uint8)


def quantize_rows(x16: np.ndarray):
    """Quantise rows of fp16 values (last axis = one (token, head) row).

    Returns (codes uint8 same shape, scales float32 shape[:-1]).
    """
    x = np.asarray(x16, dtype=np.float16).astype(np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x / scale[..., None]).astype(np.float32)
    return e4m3_encode(y), scale


def dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 values code * scale."""
    return DECODE[np.asarray(codes, dtype=np.uint8)] * np.asarray(scales, dtype=np.float64)[..., None]


# ------------------------------------------------------------------ quantised pools
# codes: uint8 per layer, [N][H][B][D] (HND) or [N][B][H][D] (NHD), the same two layouts
# as an fp16 pool; scales: float32 [N][H][B] per layer in either case.

def _rows(codes, blk, off, layout: str):
    """Index of the H code rows of slot (blk, off): codes[idx] has shape [H][D]."""
    return (blk, off) if layout == "NHD" else (blk, slice(None), off)


def append_kv(k_codes, v_codes, k_scales, v_scales, k_new, v_new, slot_mapping, block_size: int,
              layout: str = "HND") -> None:
    """Quantise token i's K/V rows (all heads) and write codes and scales to slot_mapping[i]; slot < 0 skipped."""
    kq, ks = quantize_rows(k_new)
    vq, vs = quantize_rows(v_new)
    for i, slot in enumerate(int(s) for s in slot_mapping):
        if slot < 0:
            continue
        blk, off = divmod(slot, block_size)
        k_codes[_rows(k_codes, blk, off, layout)] = kq[i]
        v_codes[_rows(v_codes, blk, off, layout)] = vq[i]
        k_scales[blk, :, off] = ks[i]
        v_scales[blk, :, off] = vs[i]


def copy_blocks(k_codes, v_codes, k_scales, v_scales, pairs) -> None:
    """Block dst <- block src in every layer, codes and scales ([L][N]... arrays)."""
    for src, dst in pairs:
        for a in (k_codes, v_codes, k_scales, v_scales):
            a[:, dst] = a[:, src]


def decode_attention(q, k_codes, v_codes, k_scales, v_scales, block_tables, context_lens, block_size: int,
                     scale=None, layout: str = "HND") -> np.ndarray:
    """Paged decode attention over a quantised layer: the float64 definition on code * scale."""
    from . import ref_attn as rf
    S, H, D = q.shape
    if scale is None:
        scale = rf.default_scale(D)
    out = np.zeros((S, H, D))
    for s in range(S):
        T = int(context_lens[s])
        if T == 0:
            continue
        blocks = [int(block_tables[s][t // block_size]) for t in range(T)]
        offs = [t % block_size for t in range(T)]
        for h in range(H):
            if layout == "NHD":
                kc, vc = k_codes[blocks, offs, h], v_codes[blocks, offs, h]
            else:
                kc, vc = k_codes[blocks, h, offs], v_codes[blocks, h, offs]
            k = dequantize(kc, k_scales[blocks, h, offs])
            v = dequantize(vc, v_scales[blocks, h, offs])
            out[s, h] = rf.attend(q[s, h], k, v, scale)
    return out
