"""DMPQ: per-layer activation precision from the block's Gamma at the previous step.

Pages: mlsanity.com "Abstract" -- a lightweight predictor gives NVFP4 to
temporally stable layers and INT8 to volatile ones, from the linear
correlation between a block's input/output difference and its layers'
quantization sensitivity; thelatestinai.com "Figure 3" -- each internal
layer fits E_rel = alpha * Gamma_{t-1} + beta; "Figure 2" -- DMPQ decides
each layer's activation bits from Gamma of the preceding step.

Readings (the pages print no decision rule):
  * the line predicts the layer's NVFP4 error; a low prediction means stable;
  * p = f32(f32(alpha * Gamma_{t-1}) + beta) in float32, no fused multiply-add;
  * NVFP4 iff p < tau (a tie goes to INT8); one global threshold tau;
  * step 0 has no previous Gamma: every layer runs INT8;
  * tau is calibrated once as the 0.6 quantile of p over an all-INT8 run so
    that about 60% of (layer, step) pairs pick NVFP4, then frozen.

Parity: pinned (tau = +inf / -inf reproduce uniform W4A4 / W4A8; alpha = 0
gives the constant decision beta < tau; step 0 -> INT8).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def predict(gamma_blocks, alpha, beta, layer_block):
    g = np.asarray(gamma_blocks, dtype=F32)[np.asarray(layer_block, dtype=np.int64)]
    ag = (np.asarray(alpha, dtype=F32) * g).astype(F32)
    return (ag + np.asarray(beta, dtype=F32)).astype(F32)


def assign(gamma_blocks, alpha, beta, layer_block, tau, step: int) -> np.ndarray:
    """uint8 flag per layer: 1 = NVFP4 activations, 0 = INT8."""
    n = len(alpha)
    if step == 0:
        return np.zeros(n, dtype=np.uint8)
    p = predict(gamma_blocks, alpha, beta, layer_block)
    return (p < F32(tau)).astype(np.uint8)


def calibrate_tau(p_values, frac: float = 0.6) -> np.float32:
    """Threshold below which `frac` of the predicted errors fall."""
    return F32(np.quantile(np.asarray(p_values, dtype=np.float64), frac))
