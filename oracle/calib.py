"""DMPQ calibration side: layer error E_rel, the Gamma -> E_rel line fit, and
the similarity of consecutive block updates.

TEST INFRASTRUCTURE ONLY (see the package header).

Pages: thelatestinai.com "Figure 1" -- per-layer relative L2 quantization
error across timesteps; "Figure 3" -- the per-layer line E_rel = alpha*Gamma +
beta fitted on the block's Gamma at the preceding step; "Figure 4" -- block
updates of consecutive steps compared by cosine similarity and relative L2
difference.  No formula is printed.  Readings:
  * E_rel(layer, t) = ||Y_q - Y||_2 / ||Y||_2 with Y = x W^T the layer's
    linear output from the unquantized bf16 input and weights, Y_q the same
    product through the quantized path (activation format of the layer,
    NVFP4 weights), both before bias / GELU / residual;
  * the line is the ordinary least-squares fit of E_rel(t) on Gamma(t-1)
    over the calibration steps t >= 1;
  * similarity of updates: cosine <a, b> / (||a|| ||b||) and relative L2
    ||a - b|| / ||b||, a the newer update.

Sums in float64 (`pair_sums`).  `pair_sums_tree` gives the same four sums
with each term rounded once in float32 (d = a - b, then d*d; b*b; a*b; a*a)
and summed by the fixed tree of oracle.gamma: the reduction the device's
pair statistics are defined by.  Parity: pinned by closed forms (exact lines
are recovered, a hand-computed three-point fit, orthogonal / parallel /
opposite vectors, identity and scaling properties of the relative error;
the tree sums within float32 rounding of the float64 ones).
"""
from __future__ import annotations

import numpy as np

from .gamma import tree_sum


def pair_sums(a, b):
    """[sum (a-b)^2, sum b^2, sum a*b, sum a^2] in float64."""
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    d = a - b
    return np.array([d @ d, b @ b, a @ b, a @ a])


def pair_sums_tree(a, b):
    """[sum (a-b)^2, sum b^2, sum a*b, sum a^2]: float32 terms, fixed tree."""
    a = np.asarray(a, dtype=np.float32).ravel()
    b = np.asarray(b, dtype=np.float32).ravel()
    d = (a - b).astype(np.float32)
    terms = ((d * d), (b * b), (a * b), (a * a))
    return np.array([tree_sum(t.astype(np.float32)) for t in terms])


def rel_l2(a, b) -> float:
    """||a - b|| / ||b|| (a the approximation of b); 0 / 0 -> 0, x / 0 -> inf."""
    s = pair_sums(a, b)
    if s[1] == 0.0:
        return 0.0 if s[0] == 0.0 else float("inf")
    return float(np.sqrt(s[0] / s[1]))


def cosine(a, b) -> float:
    """<a, b> / (||a|| ||b||); 0 when either vector is zero."""
    s = pair_sums(a, b)
    den = np.sqrt(s[3] * s[1])
    return 0.0 if den == 0.0 else float(s[2] / den)


def fit_line(x, y):
    """Least-squares alpha, beta of y ~ alpha * x + beta.  A constant x gives
    alpha = 0 and beta = mean(y)."""
    x = np.asarray(x, dtype=np.float64).ravel()
    y = np.asarray(y, dtype=np.float64).ravel()
    mx, my = x.mean(), y.mean()
    sxx = ((x - mx) ** 2).sum()
    if sxx == 0.0:
        return 0.0, float(my)
    alpha = ((x - mx) * (y - my)).sum() / sxx
    return float(alpha), float(my - alpha * mx)


def r_squared(x, y, alpha, beta) -> float:
    """Coefficient of determination of the line on (x, y); 1 when y is constant."""
    y = np.asarray(y, dtype=np.float64).ravel()
    res = y - (alpha * np.asarray(x, dtype=np.float64).ravel() + beta)
    tot = ((y - y.mean()) ** 2).sum()
    return 1.0 if tot == 0.0 else float(1.0 - (res @ res) / tot)
