"""FP8 (E4M3) KV cache: the 8-bit format written out from its definition.

[P1] "Attention that reads through the table" lists FP8 KV caches among what
production paged kernels add; [P2] "6. Квантование KV-кэша по блокам" notes
that FP8 E4M3 halves KV memory like int8 does, at practically no quality cost,
provided the scale is kept per head.

The E4M3 format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
infinities; exponent field 0 is subnormal (value = m/8 * 2^-6); the code
S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.

Readings (the pages give no more detail):
  * one fp32 scale per (layer, KV head) for K and one for V, chosen by the
    caller; a row x is stored as e4m3(fp32(x) / fp32(scale)) and stands for
    e4m3 * scale;
  * rounding to the nearest representable value, ties to even code, and
    saturation of larger magnitudes to +-448 (no NaN is ever produced from a
    finite input).
"""
from __future__ import annotations

import numpy as np


def e4m3_decode(codes) -> np.ndarray:
    """fp64 value of each uint8 E4M3 code (NaN for the two NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0, 127, dtype=np.uint8)          # +0 .. 448, strictly increasing
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x) -> np.ndarray:
    """uint8 E4M3 code of each (finite) value: nearest, ties to the even code,
    magnitudes above 448 saturate.  Works on exact fp64 inputs."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(_POS_VALUES, mag, side="left"), 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, len(_POS_VALUES) - 1)
    d_hi = np.abs(_POS_VALUES[hi] - mag)
    d_lo = np.abs(mag - _POS_VALUES[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (_POS_CODES[lo] % 2 == 0))
    code = np.where(pick_lo, _POS_CODES[lo], _POS_CODES[hi]).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)   # the sign survives rounding to 0


def quantize_rows(x, scale) -> np.ndarray:
    """Codes of rows x [T, Hkv, D] with per-head scales [Hkv]: the quotient is
    formed in fp32 (IEEE division, round to nearest), then encoded."""
    xf = np.asarray(x, dtype=np.float32)
    sf = np.asarray(scale, dtype=np.float32)
    q = (xf / sf[None, :, None]).astype(np.float32)
    return e4m3_encode(q.astype(np.float64))


def dequantize(codes, scale, head_axis: int) -> np.ndarray:
    """fp64 values codes * scale[h] with the head on `head_axis`."""
    v = e4m3_decode(codes)
    shape = [1] * v.ndim
    shape[head_axis] = -1
    return v * np.asarray(scale, dtype=np.float64).reshape(shape)
