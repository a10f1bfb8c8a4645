"""Counter-based, seeded value generator shared by the GPU path and the oracle.

This module holds no paged-attention arithmetic. It only turns integer
coordinates into reproducible pseudo-random numbers, so that the GPU side
(torch tensors on the device) and the CPU oracle (torch tensors on the host,
viewed as numpy) obtain bit-identical inputs without copying them between the
two sides.

Construction
------------
* ``mix32`` is the "lowbias32" integer hash published by Chris Wellons
  (hash-prospector): xor-shift 16, multiply by 0x7feb352d, xor-shift 15,
  multiply by 0x846ca68b, xor-shift 16, all modulo 2**32.  It is evaluated on
  int64 tensors holding values in [0, 2**32); each 32-bit product is formed
  from 16-bit halves so that no intermediate overflows int64.
* A value is the Irwin-Hall sum of four independent uniform 16-bit integers
  taken from two hash outputs, centred and scaled to unit variance:
  ``x = (u0 + u1 + u2 + u3 - 131070) * c`` with ``c = fp32(1 / 37837.227)``.
  The integer sum is exact; the single fp32 product is correctly rounded on
  every IEEE device, so host and device agree to the bit.  The distribution
  approximates N(0, 1) (mean 0, variance 1, support +-3.46).
* Rounding to the storage dtype (fp16 / bf16) is torch's round-to-nearest-even
  cast, identical on the host and on the device.
"""
from __future__ import annotations

import torch

_M32 = 0xFFFFFFFF
_C1 = 0x7FEB352D
_C2 = 0x846CA68B
# 1 / sd of the sum of four uniform integers in [0, 65535]:
# sd = 65536 * sqrt(4 / 12) * sqrt(1 - 1/65536**2) ~= 37837.227
_SCALE = float(torch.tensor(1.0 / 37837.227, dtype=torch.float32).item())
_MEAN4 = 4 * 65535 // 2  # 131070


def _mulmod32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for int64 ``x`` in [0, 2**32) without int64 overflow."""
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & _M32


def mix32(x: torch.Tensor) -> torch.Tensor:
    """lowbias32 hash of int64 values in [0, 2**32)."""
    x = x ^ (x >> 16)
    x = _mulmod32(x, _C1)
    x = x ^ (x >> 15)
    x = _mulmod32(x, _C2)
    x = x ^ (x >> 16)
    return x


def mix32_int(x: int) -> int:
    """Python-int version of :func:`mix32` (used for seeds and stream keys)."""
    x &= _M32
    x ^= x >> 16
    x = (x * _C1) & _M32
    x ^= x >> 15
    x = (x * _C2) & _M32
    x ^= x >> 16
    return x


def stream_key(seed: int, *tags: int) -> int:
    """Fold a seed and integer tags into one 32-bit stream key."""
    k = mix32_int(seed * 0x9E3779B9 + 0x632BE5AB)
    for t in tags:
        k = mix32_int(k ^ mix32_int(int(t) + 0x85EBCA6B))
    return k


def normal_from_index(key: int, idx: torch.Tensor) -> torch.Tensor:
    """fp32 approximately-N(0,1) value for every int64 counter in ``idx``.

    ``idx`` must be non-negative and below 2**62.  Works on any device.
    """
    lo = idx & _M32
    hi = idx >> 32
    a = mix32(lo ^ key)
    a = mix32(a ^ mix32(hi ^ 0x27D4EB2F))
    b = mix32(a ^ 0x165667B1)
    s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16) - _MEAN4
    return s.to(torch.float32) * _SCALE


def uniform_u32(key: int, idx: torch.Tensor) -> torch.Tensor:
    """Uniform 32-bit integers (as int64) for every counter in ``idx``."""
    lo = idx & _M32
    hi = idx >> 32
    a = mix32(lo ^ key)
    return mix32(a ^ mix32(hi ^ 0x27D4EB2F))
