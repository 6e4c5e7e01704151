"""The e4m3 8-bit float format (OCP 8-bit floating point, E4M3 variant) and the
quantisation rule of the 8-bit forward path -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.

Format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 holds
subnormals m/8 * 2^-6; exponent 15 with mantissa 7 is NaN (no infinities); the
largest finite magnitude is 1.75 * 2^8 = 448.

Quantisation ("hs-black: FlashAttention 1/2/3", section "FlashAttention-3:
precision and hardware": a scale factor per block, carried into the computation):
descale = amax / 448 in fp32 (1 for an all-zero block); code = the e4m3 value
nearest to x * (1 / descale) computed in fp32, ties to the even mantissa,
magnitudes above 448 saturating to 448, the sign kept (also on zero).
"""
from __future__ import annotations

import numpy as np


def decode(codes) -> np.ndarray:
    """fp64 values of e4m3 codes (uint8 array)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


# the 127 non-negative finite codes in increasing order of value
_POS_CODES = np.arange(0, 127, dtype=np.uint8)
_POS_VALUES = decode(_POS_CODES)


def encode(x) -> np.ndarray:
    """Nearest e4m3 code of each fp32 value (ties to the even mantissa, saturating); the sign
    bit is the sign of x, so negative values that round to zero (and -0) give -0 (0x80)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(x), 448.0)
    idx = np.searchsorted(_POS_VALUES, a)  # first value >= a
    idx = np.clip(idx, 1, 126)
    lo, hi = _POS_VALUES[idx - 1], _POS_VALUES[idx]
    pick_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((_POS_CODES[idx] & 1) == 0))
    code = np.where(pick_hi, _POS_CODES[idx], _POS_CODES[idx - 1])
    code = np.where(a == 0.0, 0, code)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def quantize_blocks(x, per_head: bool = False):
    """The 8-bit path's quantisation of x [b, s, h, d] (float array): returns
    (codes [b, s, h, d] uint8, descale fp32 [b, h, ceil(s / 128)] or [b, h])."""
    x = np.asarray(x, dtype=np.float32)
    b, s, h, d = x.shape
    nblk = (s + 127) // 128
    codes = np.zeros(x.shape, dtype=np.uint8)
    ds = np.zeros((b, h) if per_head else (b, h, nblk), dtype=np.float32)
    for bi in range(b):
        for hi in range(h):
            spans = [(0, s)] if per_head else [(k * 128, min(s, k * 128 + 128)) for k in range(nblk)]
            for k, (r0, r1) in enumerate(spans):
                blk = x[bi, r0:r1, hi, :]
                amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
                dsc = np.float32(amax) / np.float32(448.0) if amax > 0 else np.float32(1.0)
                if per_head:
                    ds[bi, hi] = dsc
                else:
                    ds[bi, hi, k] = dsc
                inv = np.float32(1.0) / np.float32(dsc)
                codes[bi, r0:r1, hi, :] = encode(blk * inv)
    if per_head:
        return codes, ds
    return codes, ds


def dequantize_blocks(codes, descale, per_head: bool = False) -> np.ndarray:
    """fp64 values codes * descale with the block layout of quantize_blocks."""
    vals = decode(codes)
    b, s, h, d = vals.shape
    ds = np.asarray(descale, dtype=np.float64)
    if per_head:
        return vals * ds[:, None, :, None]
    rows = np.arange(s) // 128
    return vals * ds[:, :, rows].transpose(0, 2, 1)[..., None]
