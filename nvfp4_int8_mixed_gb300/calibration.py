"""Offline calibration of DMPQ on the synthetic DiT stack (6Bit-Diffusion,
thelatestinai.com page: Figure 1 -- per-layer relative L2 quantization
error; Figure 3 -- the per-layer line E_rel = alpha * Gamma + beta; Figure 4
-- updates of consecutive steps compared by cosine similarity and relative
L2).

This runs once, before the denoising loop, and is not part of the
per-timestep path.  Its one product not computed by this library's kernels
is the reference Y = x W^T of E_rel, a plain fp32 library GEMM (cuBLAS
through torch.matmul, with TF32 off): the unquantized product the error is
measured against.  The quantized products, the quantizers and the pair
statistics run in the library.

The line fit is ordinary least squares of E_rel(t) on Gamma(t-1), solved
as the two-column least-squares problem [Gamma, 1] [alpha, beta]^T ~ E_rel;
its R^2 is the squared correlation of the two series.
"""
from __future__ import annotations

import numpy as np
import torch

from . import pair_stats, qlinear_w4a4, qlinear_w4a8, quantize_act_int8, quantize_act_nvfp4
from .stack import DiTStack


def fit_line(x, y):
    """(alpha, beta) minimising sum (alpha x + beta - y)^2 (float64).  With a
    constant x the slope is undetermined: alpha = 0 and beta = mean(y)."""
    x = np.asarray(x, np.float64).ravel()
    y = np.asarray(y, np.float64).ravel()
    if x.size == 0:
        raise ValueError("no calibration points")
    if np.ptp(x) == 0.0:
        return 0.0, float(np.mean(y))
    A = np.stack([x, np.ones_like(x)], axis=1)
    (alpha, beta), *_ = np.linalg.lstsq(A, y, rcond=None)
    return float(alpha), float(beta)


def r_squared(x, y) -> float:
    """Fraction of y's variance the least-squares line explains: the squared
    Pearson correlation of x and y; 1 for a constant y, 0 for a constant x."""
    x = np.asarray(x, np.float64).ravel()
    y = np.asarray(y, np.float64).ravel()
    if np.ptp(y) == 0.0:
        return 1.0
    if np.ptp(x) == 0.0:
        return 0.0
    c = np.corrcoef(x, y)[0, 1]
    return float(c * c)


def calibrate_tau(stack: DiTStack, xs, frac: float = 0.6) -> float:
    """DMPQ threshold from an all-INT8 run: the `frac` quantile of the
    predictions alpha * Gamma_{t-1} + beta over (layer, step >= 1).

    The predictions are formed on the host in float32 with the DMPQ kernel's
    rounding (f32(f32(alpha * Gamma) + beta)); choosing a quantile of them is
    a one-off calibration choice, not a per-step decision."""
    tau0, tdc0 = stack.tau, stack.max_skip
    stack.tau, stack.max_skip = float("-inf"), 0
    stack.graph = None
    stack.reset()
    _, log = stack.run(xs, record=True)
    g = torch.stack(log["gamma"][:-1]).cpu().numpy()                # Gamma_{t-1} for t = 1..T-1
    lb = stack.layer_block.cpu().numpy()
    a, b = stack.alpha.cpu().numpy(), stack.beta.cpu().numpy()
    p = (a[None, :] * g[:, lb]).astype(np.float32) + b[None, :]
    stack.tau, stack.max_skip = tau0, tdc0
    stack.graph = None
    stack.reset()
    return float(np.float32(np.quantile(p.astype(np.float64), frac)))


def calibrate_lines(stack: DiTStack, xs, weights, steps=None):
    """The calibration side of DMPQ (thelatestinai.com page, Figures 1, 3, 4)
    on the synthetic stack.

    Runs the stack eagerly with every layer in INT8 and TDC off (the same
    trajectory calibrate_tau uses).  For every step t and linear layer it
    measures E_rel = ||Y_q - Y|| / ||Y|| for both activation formats, with
    Y = x W^T in fp32 from the layer's actual bf16 input and the unquantized
    weights (a plain library GEMM: this is an offline diagnostic) and Y_q the
    W4A4 / W4A8 product of the same input.  Also per block: Gamma_t and the
    similarity of consecutive updates (cosine, relative L2).  Each layer's
    line E_rel_NVFP4(t) ~ alpha * Gamma_{b(l)}(t-1) + beta is then fitted by
    least squares over t >= 1.

    weights: the per-block dicts the stack was built from (fp32).  Returns a
    dict of numpy arrays: e_rel_nvfp4, e_rel_int8 [T, layers], gamma [T,
    blocks], delta_cos, delta_rel [T, blocks] (NaN at t = 0), alpha, beta,
    r2 [layers].
    """
    if stack.tdc_cache != "bf16":
        raise ValueError("calibration compares bf16 updates: build the stack with tdc_cache='bf16'")
    T = len(xs) if steps is None else min(steps, len(xs))
    nb = stack.nb
    names = ("qkv", "out", "up", "down")
    dev = stack.dev
    w32 = [{k: torch.as_tensor(b[k]).to(dev, torch.float32) for k in names} for b in weights]
    e4 = np.full((T, 4 * nb), np.nan)
    e8 = np.full((T, 4 * nb), np.nan)
    gam = np.zeros((T, nb))
    dcos = np.full((T, nb), np.nan)
    drel = np.full((T, nb), np.nan)
    stats = torch.empty((T, 4 * nb, 2, 4), dtype=torch.float64, device=dev)

    def hook(t):
        def measure(l, i, x):
            w = w32[l][names[i]]
            y_ref = torch.matmul(x.float(), w.t())       # fp32 library GEMM (TF32 off, see below)
            codes, sf, ga = quantize_act_nvfp4(x)
            y4 = qlinear_w4a4(codes, sf, ga, *stack.wq[l][names[i]], out_dtype=torch.float32)
            _, planes, s = quantize_act_int8(x, want_q=False)
            y8 = qlinear_w4a8(planes, s, *stack.wq[l][names[i]], out_dtype=torch.float32)
            pair_stats(y4, y_ref, out=stats[t, 4 * l + i, 0])
            pair_stats(y8, y_ref, out=stats[t, 4 * l + i, 1])
        return measure

    tau0, skip0, graph0 = stack.tau, stack.max_skip, stack.graph
    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    stack.tau, stack.max_skip, stack.graph = float("-inf"), 0, None
    stack.reset()
    prev = [None] * nb
    dstats = torch.full((T, nb, 4), float("nan"), dtype=torch.float64, device=dev)
    for t in range(T):
        stack.x_in.copy_(xs[t])
        stack.step_dev.fill_(t)
        old = [d.clone() for d in stack.delta] if t >= 1 else None
        stack.enqueue_step(hook=hook(t))
        if old is not None:                        # Delta_{t-1} existed: compare Delta_t with it
            for l in range(nb):
                pair_stats(stack.delta[l], old[l], out=dstats[t, l])
        gam[t] = stack.gamma.cpu().numpy()
    torch.cuda.synchronize()
    st = stats.cpu().numpy()
    with np.errstate(divide="ignore", invalid="ignore"):
        e4[:] = np.sqrt(st[:, :, 0, 0] / st[:, :, 0, 1])
        e8[:] = np.sqrt(st[:, :, 1, 0] / st[:, :, 1, 1])
        ds = dstats.cpu().numpy()
        drel[:] = np.sqrt(ds[:, :, 0] / ds[:, :, 1])
        dcos[:] = ds[:, :, 2] / np.sqrt(ds[:, :, 3] * ds[:, :, 1])
    lb = stack.layer_block.cpu().numpy()
    alpha = np.zeros(4 * nb)
    beta = np.zeros(4 * nb)
    r2 = np.zeros(4 * nb)
    for k in range(4 * nb):
        x = gam[:T - 1, lb[k]]                     # Gamma_{t-1}
        y = e4[1:T, k]                             # E_rel at t
        alpha[k], beta[k] = fit_line(x, y)
        r2[k] = r_squared(x, y)
    stack.tau, stack.max_skip, stack.graph = tau0, skip0, graph0
    torch.backends.cuda.matmul.allow_tf32 = tf32
    stack.reset()
    return dict(e_rel_nvfp4=e4, e_rel_int8=e8, gamma=gam, delta_cos=dcos, delta_rel=drel, alpha=alpha, beta=beta,
                r2=r2)
