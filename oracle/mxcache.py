"""Compressed TDC cache (an extension, not from the pages): the block update
Delta stored as E4M3 codes with one power-of-two scale per 32 elements.

TEST INFRASTRUCTURE ONLY (see the package header).

Pages: TDC reuses a block's update from the preceding steps ("Figure 2",
thelatestinai.com page); nothing about how it is stored.  At video-DiT sizes
one bf16 update per block is 2 GB (2B model) to 9 GB (5B with CFG).  The
reading here halves that:
  * block b = elements 32b .. 32b+31 of the flattened tensor (n % 32 == 0);
  * A_b = max |v_i| over the block (bf16 values, exact in float32);
  * scale exponent k_b = the smallest integer with A_b <= 448 * 2^k_b,
    clamped to [-127, 127]; k_b = -127 when A_b = 0; stored as the byte
    k_b + 127;
  * code_i = E4M3(v_i * 2^-k_b), round to nearest even, saturating (the
    product is exact);
  * decoded value = E4M3(code_i) * 2^k_b (exact in float32).
Layout: n code bytes, then n/32 scale bytes.  Element type and block size
are those of the OCP microscaling MXFP8 (E4M3) format; its shared-exponent
rule, floor(log2 A_b) - 8, can clip a block's largest element by up to
12.5 %, and this rule never clips.

Parity: pinned (values on the grid round-trip, the scale boundary at
A_b = 448 * 2^k, zero blocks, the half-step error bound, nearest code by
brute force through the E4M3 table, byte layout).
"""
from __future__ import annotations

import numpy as np

from .codecs import bf16_to_f32, e4m3_decode, e4m3_encode

BLOCK = 32
E4M3_MAX = 448.0


def scale_exponent(amax) -> np.ndarray:
    """k_b for block maxima A_b >= 0 (float array): smallest k with A <= 448 * 2^k."""
    a = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(a)                          # a = m * 2^e, m in [0.5, 1)
    # a = (2m) * 2^(e-1) with 2m in [1, 2); 448 * 2^k = 1.75 * 2^(k+8)
    k = (e - 1) - 8 + (2.0 * m > 1.75)
    k = np.where(a == 0, -127, k)
    return np.clip(k, -127, 127).astype(np.int64)


def encode(v):
    """float32 values (bf16-valued), n % 32 == 0 -> (codes uint8 [n], scale bytes uint8 [n/32])."""
    v = np.asarray(v, dtype=np.float32).reshape(-1)
    assert v.size % BLOCK == 0
    blocks = v.astype(np.float64).reshape(-1, BLOCK)
    k = scale_exponent(np.max(np.abs(blocks), axis=1))
    scaled = blocks * np.exp2(-k.astype(np.float64))[:, None]       # exact: power-of-two scaling
    codes = e4m3_encode(scaled.astype(np.float32).reshape(-1))
    return codes, (k + 127).astype(np.uint8)


def decode(codes, scales) -> np.ndarray:
    """(codes [n], scale bytes [n/32]) -> float32 [n]."""
    c = e4m3_decode(np.asarray(codes, dtype=np.uint8)).astype(np.float64).reshape(-1, BLOCK)
    k = np.asarray(scales, dtype=np.uint8).astype(np.int64) - 127
    return (c * np.exp2(k.astype(np.float64))[:, None]).astype(np.float32).reshape(-1)


def to_bytes(codes, scales) -> np.ndarray:
    """The device layout: codes, then scale bytes."""
    return np.concatenate([np.asarray(codes, np.uint8).reshape(-1), np.asarray(scales, np.uint8).reshape(-1)])


def roundtrip_bf16(delta_bits) -> np.ndarray:
    """The cached value of a bf16 update: decode(encode(Delta)) as float32 (same shape)."""
    d = bf16_to_f32(delta_bits)
    return decode(*encode(d)).reshape(d.shape)
