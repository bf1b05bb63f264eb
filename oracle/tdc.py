"""TDC: Temporal Delta Cache -- skip a block whose update barely changes.

Pages: mlsanity.com "Abstract" -- the residual between a transformer block's
input and output is temporally consistent, so TDC skips the computation of
these invariant blocks; thelatestinai.com "Figure 2" -- the skip is decided
from the block updates Delta of the preceding two steps; "Figure 4" --
updates are compared by cosine similarity and relative L2 difference.

Readings (no rule is printed):
  * the cache keeps the most recent *computed* update Delta_fresh of each
    block (bf16), the relative change r2 measured when it was produced
    (against the update before it) and two counters;
  * skip at step t  <=>  fresh_count >= 2  and  r2 < f32(tau_tdc^2)
                          and  consec < max_skip      (max_skip = 1 by default,
    so a skipped step is followed by a computed one and a reused update never
    compounds);
  * a skipped block outputs bf16(f32(in) + f32(Delta_fresh)); its cache is
    unchanged except consec + 1;
  * a computed block stores its new update, measures r2 against the old one
    (if any), fresh_count + 1, consec = 0.

PDR ("Table 3" names it as a component; the pages give no definition).
Variants of the reading above, each a parameter of the same rule:
  * "purified" Delta: Delta is replaced only by a computed step, so a reused
    update never feeds the next one (the default above);
  * max_skip > 1: up to max_skip consecutive reuses;
  * periodic refresh: with refresh_every = k > 0, a step t with t % k == 0 is
    always computed, whatever r2 says.

Parity: pinned (tau_tdc = 0 never skips; max_skip = 0 never skips; a forced
skip gives out - in equal to Delta up to one bf16 rounding; hand-written r2
sequences give hand-derived skip patterns, also with max_skip = 2 and a
periodic refresh).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .codecs import bf16_to_f32, f32_to_bf16

F32 = np.float32


@dataclass
class BlockCache:
    fresh_count: int = 0
    consec: int = 0
    r2: np.float32 = F32(np.inf)
    delta: np.ndarray | None = None       # bf16 bits, or float32 cached values (compressed cache)


def decide(cache: BlockCache, tau_tdc: float, max_skip: int, refresh_every: int = 0, step: int = 0) -> bool:
    if refresh_every > 0 and step % refresh_every == 0:
        return False                       # periodic refresh: this step is computed
    t2 = F32(F32(tau_tdc) * F32(tau_tdc))
    return cache.fresh_count >= 2 and F32(cache.r2) < t2 and cache.consec < max_skip


def apply(xin, delta_fresh):
    """Skipped block output: bf16(f32(in) + f32(Delta_fresh)); Delta_fresh is bf16
    bits or the float32 value of a compressed cache."""
    d = np.asarray(delta_fresh)
    df = bf16_to_f32(d) if d.dtype == np.uint16 else d.astype(F32)
    return f32_to_bf16((bf16_to_f32(xin) + df).astype(F32))


def after_skip(cache: BlockCache) -> None:
    cache.consec += 1


def after_compute(cache: BlockCache, delta_new, r2) -> None:
    cache.delta = delta_new
    if r2 is not None:
        cache.r2 = F32(r2)
    cache.fresh_count += 1
    cache.consec = 0
