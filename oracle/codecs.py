"""Number formats: E2M1 (FP4), E4M3 (FP8) and bf16, written from their definitions.

The 6Bit-Diffusion pages name NVFP4 (abstract, mlsanity.com page) but print
no format.  The formats here follow the OCP definitions:
  * E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; magnitudes
    {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no Inf/NaN.
  * E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
    subnormals m * 2^-9; max 448; 0x7F/0xFF are NaN; no Inf.
Encoding is round-to-nearest, ties to the even code, saturating to the
largest finite magnitude.  A value that rounds to zero keeps its sign
(-0.1 -> E2M1 code 0x8).  These are the semantics of the
`cvt.rn.satfinite.{e2m1x2,e4m3x2}.f32` conversions the GPU path uses; they
were checked on the device for every tie listed in the tests.

Encoders are brute force: distance to every finite grid value, nearest wins.
Parity: pinned (grid tables, ties, saturation; E4M3 also against torch's
float8_e4m3fn conversion).
"""
from __future__ import annotations

import numpy as np

# ------------------------------------------------------------------ E2M1
def e2m1_decode(code) -> np.ndarray:
    """4-bit code(s) -> float32 value(s)."""
    c = np.asarray(code).astype(np.int64) & 0xF
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return np.where(s == 1, -mag, mag).astype(np.float32)


_E2M1_MAG = e2m1_decode(np.arange(8)).astype(np.float64)  # index = code & 7


def e2m1_encode(v) -> np.ndarray:
    """float32 value(s) -> 4-bit code(s) (uint8), RNE, satfinite, signed zero."""
    v = np.asarray(v, dtype=np.float32)
    flat = v.reshape(-1).astype(np.float64)
    a = np.abs(flat)
    dist = np.abs(a[:, None] - _E2M1_MAG[None, :])          # [n, 8]
    best = dist.min(axis=1)
    idx = np.argmin(dist, axis=1)                            # lowest index among ties
    tie = (dist == best[:, None]).sum(axis=1) > 1
    idx = np.where(tie & (idx % 2 == 1), idx + 1, idx)       # tie -> even code
    idx = np.where(a >= 6.0, 7, idx)                         # saturate
    neg = np.signbit(flat)
    code = (idx + np.where(neg, 8, 0)).astype(np.uint8)
    return code.reshape(v.shape)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[R, K] 4-bit codes -> [R, K/2] bytes; element 2j in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ------------------------------------------------------------------ E4M3
def e4m3_decode(code) -> np.ndarray:
    """8-bit code(s) -> float32 value(s) (NaN for 0x7F/0xFF)."""
    c = np.asarray(code).astype(np.int64) & 0xFF
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag).astype(np.float32)


_E4M3_MAG = e4m3_decode(np.arange(0x7F)).astype(np.float64)  # codes 0x00..0x7E, increasing


def e4m3_encode(v) -> np.ndarray:
    """float32 value(s) -> E4M3 code(s) (uint8), RNE, satfinite, signed zero."""
    v = np.asarray(v, dtype=np.float32)
    flat = v.reshape(-1).astype(np.float64)
    a = np.abs(flat)
    hi = np.searchsorted(_E4M3_MAG, a, side="left").clip(0, len(_E4M3_MAG) - 1)
    lo = (hi - 1).clip(0, None)
    dlo = np.abs(a - _E4M3_MAG[lo])
    dhi = np.abs(_E4M3_MAG[hi] - a)
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= _E4M3_MAG[-1], len(_E4M3_MAG) - 1, pick)   # saturate at 448
    neg = np.signbit(flat)
    code = (pick + np.where(neg, 0x80, 0)).astype(np.uint8)
    return code.reshape(v.shape)


# ------------------------------------------------------------------ bf16
def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (finite inputs)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def f64_to_bf16(x) -> np.ndarray:
    """float64 -> float32 (RNE) -> bf16 (RNE): the kernels' output path."""
    return f32_to_bf16(np.asarray(x, dtype=np.float64).astype(np.float32))
