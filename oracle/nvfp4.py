"""NVFP4 quantization of an activation (or weight) tensor.

Pages: the mlsanity.com "Abstract" gives NVFP4 to temporally stable layers;
nothing else about the format is printed.  Reading (stated, not from the
pages): NVFP4 = E2M1 codes, one E4M3 scale S per 16 consecutive elements
along K, one float32 tensor scale g.  Steps, all float32 round-to-nearest:

  1. amax_t = max |x| over the tensor (or the caller's value);
  2. g = amax_t / 2688 (2688 = 6 * 448, the largest E2M1 times the largest
     E4M3 magnitude); g = 1 when amax_t = 0;
  3. per 16-element block b: amax_b = max |x| over the block;
  4. s_b = (amax_b * 448) / amax_t  (the product is exact; s_b = 0 when
     amax_t = 0);  S_b = E4M3(s_b);
  5. d_b = S_b * g; if d_b = 0 every code of the block is +0; otherwise
     r_b = 1 / d_b and code_k = E2M1(x_k * r_b);
  6. pack two codes per byte, element 2j in the low nibble.
The value a code stands for is E2M1(code) * S_b * g.

Scale-factor layout for the tensor-core consumer (reading: the 1-D block
scaling layout of the Blackwell block-scaled MMA): rows are padded to a
multiple of 128 and the K/16 scale columns to a multiple of 4; the byte of
row m, scale column c sits at
    ((m // 128) * (Kc4 // 4) + c // 4) * 512 + (m % 32) * 16 + ((m % 128) // 32) * 4 + c % 4
with Kc4 the padded column count.  Pads are zero.

Delayed scaling (an extension for quantizing inside the producing kernel,
not from the pages): a producer that emits NVFP4 in one pass cannot know the
tensor amax of what it is producing.  It uses instead headroom * (the exact
tensor amax of the same layer input at the previous call), and records this
call's exact amax for the next one.  With a power-of-two headroom the
product S_b * g is unchanged whenever the amax did not grow (S_b halves and g
doubles exactly, E4M3 subnormals aside), so the headroom costs no precision;
an amax that grew past headroom * previous saturates the largest blocks at
+-6 * 448 * g = +-amax_used.  `quantize_delayed` is steps 1-6 with amax_t =
headroom * amax_prev.

Parity: pinned (hand-built blocks with known scales, brute-force nearest
code, swizzle bijection and fixed offsets; delayed scaling by the zero
history, the power-of-two identity and the saturation bound).
"""
from __future__ import annotations

import numpy as np

from .codecs import e2m1_encode, e4m3_encode, e4m3_decode, pack_e2m1, unpack_e2m1, e2m1_decode

F32 = np.float32
E2M1_MAX = 6.0
E4M3_MAX = 448.0


def tensor_amax(x: np.ndarray) -> np.float32:
    return F32(np.max(np.abs(x.astype(F32)))) if x.size else F32(0.0)


def global_scale(amax_t) -> np.float32:
    amax_t = F32(amax_t)
    if amax_t == 0:
        return F32(1.0)
    return F32(amax_t / F32(E2M1_MAX * E4M3_MAX))


def quantize(x: np.ndarray, amax_t=None):
    """x: float32 [R, K] (bf16 values), K % 16 == 0.

    Returns (packed codes uint8 [R, K/2], scale bytes uint8 [R, K/16], g float32, amax_t).
    """
    x = np.asarray(x, dtype=F32)
    R, K = x.shape
    assert K % 16 == 0
    if amax_t is None:
        amax_t = tensor_amax(x)
    amax_t = F32(amax_t)
    g = global_scale(amax_t)
    xb = x.reshape(R, K // 16, 16)
    amax_b = np.max(np.abs(xb), axis=2).astype(F32)                       # [R, K/16]
    if amax_t == 0:
        s = np.zeros_like(amax_b)
    else:
        s = ((amax_b * F32(E4M3_MAX)).astype(F32) / amax_t).astype(F32)
    sf = e4m3_encode(s)                                                    # [R, K/16]
    S = e4m3_decode(sf)
    d = (S * g).astype(F32)
    nz = d != 0
    r = np.zeros_like(d)
    r[nz] = (F32(1.0) / d[nz]).astype(F32)
    v = (xb * r[:, :, None]).astype(F32)
    codes = e2m1_encode(v)
    codes = np.where(nz[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    return pack_e2m1(codes.reshape(R, K)), sf.astype(np.uint8), g, amax_t


def quantize_delayed(x: np.ndarray, amax_prev, headroom=2.0):
    """Delayed-scaling NVFP4: quantize with amax_t = f32(headroom * amax_prev).

    Returns (codes, scale bytes, g, amax_used, amax_new) with amax_new the
    exact tensor amax of x, the history value for the next call."""
    amax_used = F32(F32(headroom) * F32(amax_prev))
    codes, sf, g, _ = quantize(x, amax_used)
    return codes, sf, g, amax_used, tensor_amax(x)


def dequantize(packed: np.ndarray, sf: np.ndarray, g=1.0) -> np.ndarray:
    """Codes and scale bytes -> float64 [R, K] values E2M1 * S * g."""
    codes = unpack_e2m1(packed)
    R, K = codes.shape
    vals = e2m1_decode(codes).astype(np.float64).reshape(R, K // 16, 16)
    S = e4m3_decode(sf).astype(np.float64)
    return (vals * S[:, :, None]).reshape(R, K) * float(g)


# ------------------------------------------------------------ SF layout
def sf_padded_shape(R: int, K: int):
    kc = K // 16
    return (R + 127) // 128 * 128, (kc + 3) // 4 * 4


def sf_offset(m, c, kc4: int):
    m = np.asarray(m, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    return ((m // 128) * (kc4 // 4) + c // 4) * 512 + (m % 32) * 16 + ((m % 128) // 32) * 4 + c % 4


def swizzle_sf(sf: np.ndarray) -> np.ndarray:
    """Plain [R, K/16] scale bytes -> flat swizzled buffer with zero pads."""
    R, kc = sf.shape
    rp, kc4 = sf_padded_shape(R, kc * 16)
    out = np.zeros(rp * kc4, dtype=np.uint8)
    m, c = np.meshgrid(np.arange(R), np.arange(kc), indexing="ij")
    out[sf_offset(m, c, kc4)] = sf
    return out


def unswizzle_sf(buf: np.ndarray, R: int, K: int) -> np.ndarray:
    rp, kc4 = sf_padded_shape(R, K)
    kc = K // 16
    m, c = np.meshgrid(np.arange(R), np.arange(kc), indexing="ij")
    return np.asarray(buf, dtype=np.uint8).reshape(-1)[sf_offset(m, c, kc4)]
