"""Per-token symmetric INT8 activation quantization.

Pages: the mlsanity.com "Abstract" keeps INT8 for volatile layers; the
granularity and rounding are not printed.  Reading: one scale per token
(row), symmetric, round to nearest even, clamp to [-127, 127] (-128 is never
produced).  float32 arithmetic:

  amax_m = max |x| over row m (or the caller's value);
  amax_m = 0  ->  the row's codes are 0 and s_m = 0;
  otherwise inv = 127 / amax_m,  q = clamp(rne(x * inv), -127, 127),
            s_m = amax_m / 127.
The value a code stands for is q * s_m.

Also here: the exact base-8 digit split of an INT8 code that lets the
tensor-core GEMM consume INT8 activations as three E2M1 digit planes
(q = 64 a + 8 b + c, each digit an integer E2M1 value).  This is an
identity on integers, not a quantization step; it is checked against q.

Parity: pinned (+-amax -> +-127, zero row, saturation, ties to even; digit
split reconstructs every q in [-127, 127]).
"""
from __future__ import annotations

import numpy as np

from .codecs import e2m1_encode

F32 = np.float32


def row_amax(x: np.ndarray) -> np.ndarray:
    return np.max(np.abs(np.asarray(x, dtype=F32)), axis=1).astype(F32)


def quantize(x: np.ndarray, amax=None):
    """x float32 [R, K] -> (q int8 [R, K], s float32 [R], amax float32 [R])."""
    x = np.asarray(x, dtype=F32)
    amax = row_amax(x) if amax is None else np.asarray(amax, dtype=F32).reshape(-1)
    nz = amax > 0
    inv = np.zeros_like(amax)
    inv[nz] = (F32(127.0) / amax[nz]).astype(F32)
    v = (x * inv[:, None]).astype(F32)
    q = np.clip(np.rint(v), -127, 127).astype(np.int8)
    q[~nz, :] = 0
    s = np.zeros_like(amax)
    s[nz] = (amax[nz] / F32(127.0)).astype(F32)
    return q, s, amax


def digits(q: np.ndarray):
    """Split int8 codes into three integer digits (a, b, c), q = 64a + 8b + c.

    c is q mod 8 taken in [-3, 4]; b likewise for (q - c) / 8; a = the rest,
    in [-2, 2].  Every digit is an integer E2M1 value (0, +-1, +-2, +-3, +-4).
    """
    q = np.asarray(q, dtype=np.int64)
    c = q % 8
    c = np.where(c > 4, c - 8, c)
    q1 = (q - c) // 8
    b = q1 % 8
    b = np.where(b > 4, b - 8, b)
    a = (q1 - b) // 8
    return a, b, c


def digit_codes(q: np.ndarray):
    """E2M1 codes of the three digit planes of q (uint8, unpacked)."""
    a, b, c = digits(q)
    return tuple(e2m1_encode(d.astype(F32)) for d in (a, b, c))
