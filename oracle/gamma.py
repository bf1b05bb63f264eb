"""Gamma (block relative L1 input/output distance), the block update Delta and
the TDC change metric.

TEST INFRASTRUCTURE ONLY (see the package header).

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

Summation (a reading: the pages fix no precision).  Gamma and r2 decide
DMPQ flags and TDC skips, so their bits must not depend on how a machine
schedules the sum.  They are defined by one fixed reduction tree:
  * per-element terms in float32, round to nearest: d = f32(out) - f32(in),
    |d| and |in| for Gamma; e = f32(Delta_new) - f32(Delta_prev), e*e and
    Delta_prev*Delta_prev (each product rounded once) for r2;
  * the flat tensor is cut into tiles of 8192 elements (the last one
    partial; missing elements contribute nothing);
  * inside a tile, element j*2048 + 8*t + e (j = 0..3, t = 0..255,
    e = 0..7) belongs to lane t; a lane adds its 32 terms one at a time in
    increasing element order, in float32;
  * the 256 lane sums of a tile are combined pairwise in float32: first
    lanes t and t^16, then t^8, t^4, t^2, t^1 (a butterfly inside each group
    of 32 lanes), then the eight group sums g by g[w] + g[w + 4], then
    + g[w + 2], then + g[w + 1];
  * tile sums are widened to float64; lane k (k = 0..255) adds the tiles
    k, k + 256, k + 512, ... in order, then the 256 lane sums are combined
    by halving (s[k] + s[k + 128], then + 64, ..., + 1);
  * Gamma = f32(S1 / S0) and r2 = f32(Sd / So), each a float64 division
    rounded once to float32.
All terms are >= 0, so the tree's result lies within a few float32
roundings of the exact sum (`gamma_exact`, `rel_l2_sq_exact` give the
textbook float64 values the tests bound it against).

With the compressed cache (oracle.mxcache, an extension) the previous update
is the cached value decode(encode(Delta_prev)) and the pass stores
encode(Delta_new); r2 compares the exact bf16 Delta_new with that cached
value.

Parity: pinned (out = in -> 0; out = 2 in -> 1; Delta_new = Delta_prev -> 0;
Delta_new = 2 Delta_prev -> 1; a tile of ones sums to 8192; the tree agrees
with a scalar walk of the same tree on small ragged inputs and with the
exact float64 sums within its rounding bound).
"""
from __future__ import annotations

import numpy as np

from . import mxcache
from .codecs import bf16_to_f32, f32_to_bf16

F32 = np.float32
TILE = 8192
LANES = 256
VEC = 8                       # consecutive elements a lane takes at a time
STEPS = TILE // (LANES * VEC)  # 4 groups of 8 per lane and tile


def tree_sum(terms) -> np.float64:
    """Sum of float32 terms by the fixed tree of the module header."""
    t = np.asarray(terms, dtype=F32).ravel()
    n = t.size
    ntiles = max(1, -(-n // TILE))
    padded = np.zeros(ntiles * TILE, dtype=F32)
    padded[:n] = t
    x = padded.reshape(ntiles, STEPS, LANES, VEC)             # [tile, j, lane, e]
    lane = np.zeros((ntiles, LANES), dtype=F32)
    for j in range(STEPS):
        for e in range(VEC):
            lane = (lane + x[:, j, :, e]).astype(F32)
    g = lane.reshape(ntiles, LANES // 32, 32)
    idx = np.arange(32)
    for h in (16, 8, 4, 2, 1):
        g = (g + g[:, :, idx ^ h]).astype(F32)
    w = g[:, :, 0].copy()                                     # [tile, 8] group sums
    for h in (4, 2, 1):
        w[:, :h] = (w[:, :h] + w[:, h:2 * h]).astype(F32)
    tiles = w[:, 0].astype(np.float64)
    nb = -(-ntiles // LANES)
    tp = np.zeros(nb * LANES, dtype=np.float64)
    tp[:ntiles] = tiles
    acc = np.zeros(LANES, dtype=np.float64)
    for b in range(nb):
        acc = acc + tp[b * LANES:(b + 1) * LANES]
    h = LANES // 2
    while h >= 1:
        acc[:h] = acc[:h] + acc[h:2 * h]
        h //= 2
    return np.float64(acc[0])


def _ratio(num: np.float64, den: np.float64, zero_den) -> np.float32:
    return zero_den if den == 0.0 else F32(np.float64(num) / np.float64(den))


def gamma(xin, xout) -> np.float32:
    fi = bf16_to_f32(xin).astype(F32).ravel()
    d = (bf16_to_f32(xout).astype(F32).ravel() - fi).astype(F32)
    return _ratio(tree_sum(np.abs(d)), tree_sum(np.abs(fi)), F32(0.0))


def delta(xin, xout):
    """Stored update bf16(f32(out) - f32(in)) as bf16 bits."""
    d = (bf16_to_f32(xout) - bf16_to_f32(xin)).astype(F32)
    return f32_to_bf16(d)


def _f32(d):
    """bf16 bits (uint16) or float32 values -> float32."""
    d = np.asarray(d)
    return (bf16_to_f32(d) if d.dtype == np.uint16 else d.astype(F32)).astype(F32).ravel()


def rel_l2_sq(delta_new, delta_prev) -> np.float32:
    dn = _f32(delta_new)
    dp = _f32(delta_prev)
    e = (dn - dp).astype(F32)
    sd = tree_sum((e * e).astype(F32))
    so = tree_sum((dp * dp).astype(F32))
    return _ratio(sd, so, F32(np.inf))


def gamma_exact(xin, xout) -> float:
    """Textbook value: float64 sums of the exact float64 terms."""
    fi = bf16_to_f32(xin).astype(np.float64)
    fo = bf16_to_f32(xout).astype(np.float64)
    s0 = np.sum(np.abs(fi))
    return 0.0 if s0 == 0 else float(np.sum(np.abs(fo - fi)) / s0)


def rel_l2_sq_exact(delta_new, delta_prev) -> float:
    dn = _f32(delta_new).astype(np.float64)
    dp = _f32(delta_prev).astype(np.float64)
    so = np.sum(dp * dp)
    return float("inf") if so == 0 else float(np.sum((dn - dp) ** 2) / so)


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
