"""Gamma (block relative L1 input/output distance), the block update Delta and
the TDC change metric.

Pages (thelatestinai.com): "Figure 2" -- Gamma is the block's input/output
relative L1 distance at the preceding step; "Figure 3" -- Gamma_{t-1}
drives each internal layer's line; "Figure 4" -- the block update
Delta = out - in is compared between adjacent steps by cosine similarity and
relative L2 difference.

Definitions (reading: norms over the whole block tensor, all tokens):
  Gamma   = ||out - in||_1 / ||in||_1                   (0 when ||in||_1 = 0)
  Delta   = bf16(f32(out) - f32(in))                    (float32 subtraction,
            then round to bf16: the stored update)
  r2      = ||Delta_new - Delta_prev||_2^2 / ||Delta_prev||_2^2
            (older update in the denominator; +inf when it is 0)
  cos     = <Delta_new, Delta_prev> / (||Delta_new|| ||Delta_prev||)
Sums are float64 over exact float64 values of the bf16 inputs; the ratio is
rounded to float32.

With the compressed cache (oracle.mxcache, an extension) the previous update
is the cached value decode(encode(Delta_prev)) and the pass stores
encode(Delta_new); r2 compares the exact bf16 Delta_new with that cached
value.

Parity: pinned (out = in -> 0; out = 2 in -> 1; Delta_new = Delta_prev -> 0;
Delta_new = 2 Delta_prev -> 1; constant tensors in closed form).
"""
from __future__ import annotations

import numpy as np

from . import mxcache
from .codecs import bf16_to_f32, f32_to_bf16

F32 = np.float32


def gamma(xin, xout) -> np.float32:
    fi = bf16_to_f32(xin).astype(np.float64)
    fo = bf16_to_f32(xout).astype(np.float64)
    s0 = np.sum(np.abs(fi))
    s1 = np.sum(np.abs(fo - fi))
    return F32(0.0) if s0 == 0 else F32(s1 / s0)


def delta(xin, xout):
    """Stored update bf16(f32(out) - f32(in)) as bf16 bits."""
    d = (bf16_to_f32(xout) - bf16_to_f32(xin)).astype(F32)
    return f32_to_bf16(d)


def _f64(d):
    """bf16 bits (uint16) or float32 values -> float64."""
    d = np.asarray(d)
    return (bf16_to_f32(d) if d.dtype == np.uint16 else d.astype(np.float32)).astype(np.float64)


def rel_l2_sq(delta_new, delta_prev) -> np.float32:
    dn = _f64(delta_new)
    dp = _f64(delta_prev)
    so = np.sum(dp * dp)
    sd = np.sum((dn - dp) ** 2)
    return F32(np.inf) if so == 0 else F32(sd / so)


def cosine(delta_new, delta_prev) -> float:
    dn = bf16_to_f32(delta_new).astype(np.float64).ravel()
    dp = bf16_to_f32(delta_prev).astype(np.float64).ravel()
    den = np.linalg.norm(dn) * np.linalg.norm(dp)
    return 0.0 if den == 0 else float(dn @ dp / den)


def block_pass(xin, xout, delta_prev=None, computed=True, cache="bf16"):
    """One pass of the kernel's contract.

    Returns (Gamma, Delta_new or None, r2 or None).  Delta_new is produced
    only for a computed block; r2 only when a previous update exists.
    cache "bf16": Delta_new is the bf16 update (bits); "mx": the cached value
    decode(encode(Delta_new)) as float32, and delta_prev is such a value.
    """
    g = gamma(xin, xout)
    if not computed:
        return g, None, None
    dn = delta(xin, xout)
    r2 = None if delta_prev is None else rel_l2_sq(dn, delta_prev)
    if cache == "mx":
        dn = mxcache.roundtrip_bf16(dn)
    return g, dn, r2
