"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module only draws random numbers and stores them in the activation
dtype (bf16, kept as raw uint16 bit patterns).  It holds none of the
quantization method's arithmetic: no scales, no codes, no reductions.

Workload shapes follow the video-DiT settings the 6Bit-Diffusion pages
evaluate on (CogVideoX-2B/5B, "Table 1" and "Table 2" of the
thelatestinai.com page); the trained models and VBench prompts are not
available, so normally distributed activations with a few outlier channels
and N(0, 0.02) weights stand in for them.

All generators use numpy's PCG64 bit generator with an explicit seed.
"""
from __future__ import annotations

import numpy as np

# 2B-class token count: 13 latent frames x 30 x 45 patches + 226 text tokens.
M_2B = 13 * 30 * 45 + 226  # 17776


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def activations(g: np.random.Generator, M: int, K: int, n_outliers: int,
                lo: float, hi: float | None = None) -> np.ndarray:
    """N(0,1) activations [M,K] with `n_outliers` channels scaled up.

    With `hi` None every outlier channel is scaled by `lo`; otherwise each gets
    its own factor drawn from U(lo, hi).  Returns bf16 bits [M,K].
    """
    x = g.standard_normal((M, K), dtype=np.float32)
    if n_outliers > 0:
        cols = g.choice(K, n_outliers, replace=False)
        if hi is None:
            fac = np.full(n_outliers, lo, dtype=np.float32)
        else:
            fac = g.uniform(lo, hi, n_outliers).astype(np.float32)
        x[:, cols] *= fac[None, :]
    return f32_to_bf16_bits(x)


def weights(g: np.random.Generator, N: int, K: int, std: float = 0.02) -> np.ndarray:
    """N(0, std) weights stored out x in ([N,K], K contiguous) as float32."""
    return (g.standard_normal((N, K), dtype=np.float32) * np.float32(std)).astype(np.float32)


def bias(g: np.random.Generator, N: int, std: float = 0.02) -> np.ndarray:
    return f32_to_bf16_bits(g.standard_normal(N, dtype=np.float32) * np.float32(std))


# ---------------------------------------------------------------- config 1
def tiny_layer(seed: int = 0):
    """Single 256x256 activation, 4 outlier channels x20; weight 256x512 (KxN)
    transposed to [N=512, K=256]; a Gamma pair out = in + 0.05 N(0,1)."""
    g = rng(seed)
    a = activations(g, 256, 256, 4, 20.0)
    w_kn = g.standard_normal((256, 512), dtype=np.float32) * np.float32(0.02)
    w = np.ascontiguousarray(w_kn.T)
    b = bias(g, 512)
    res = f32_to_bf16_bits(g.standard_normal((256, 512), dtype=np.float32))
    gin = a
    gout = f32_to_bf16_bits(bf16_bits_to_f32(gin) + np.float32(0.05) * g.standard_normal((256, 256), dtype=np.float32))
    return dict(a=a, w=w, bias=b, residual=res, gamma_in=gin, gamma_out=gout)


# ------------------------------------------------------------ configs 2, 3
GEMM_SHAPES = {
    # name: (K, N, epilogue) -- epilogue as (gelu, residual)
    "2B": [("qkv", 1920, 5760, False, False), ("out_proj", 1920, 1920, False, True),
           ("ffn_up", 1920, 7680, True, False), ("ffn_down", 7680, 1920, False, True)],
    "5B": [("qkv", 3072, 9216, False, False), ("out_proj", 3072, 3072, False, True),
           ("ffn_up", 3072, 12288, True, False), ("ffn_down", 12288, 3072, False, True)],
}


def gemm_layer(seed: int, M: int, K: int, N: int, residual: bool):
    """One layer of the 2B/5B GEMM sets: A N(0,1) with 1% of channels x U(10,50),
    W N(0,0.02) [N,K], zero bias, optional N(0,1) residual [M,N]."""
    g = rng(seed)
    a = activations(g, M, K, max(1, int(0.01 * K)), 10.0, 50.0)
    w = weights(g, N, K)
    r = f32_to_bf16_bits(g.standard_normal((M, N), dtype=np.float32)) if residual else None
    return dict(a=a, w=w, residual=r)


def gamma_pair(seed: int, M: int, H: int, scale: float = 0.05):
    """Block input/output pair for the Gamma/Delta pass: out = in + scale*N(0,1),
    plus a previous fresh Delta of similar magnitude."""
    g = rng(seed)
    xin = f32_to_bf16_bits(g.standard_normal((M, H), dtype=np.float32))
    xin_f = bf16_bits_to_f32(xin)
    d0 = g.standard_normal((M, H), dtype=np.float32) * np.float32(scale)
    xout = f32_to_bf16_bits(xin_f + d0)
    dprev = f32_to_bf16_bits(d0 + np.float32(scale * 0.1) * g.standard_normal((M, H), dtype=np.float32))
    return dict(xin=xin, xout=xout, delta_prev=dprev)


# ------------------------------------------------------------ configs 4, 5
def stack_setup(seed: int, n_blocks: int, H: int, F: int):
    """Weights of a synthetic DiT block stack and the per-layer predictor lines.

    Each block has 4 linear layers in this order: qkv [3H,H], out [H,H],
    up [F,H], down [H,F].  (alpha, beta) per layer ~ U(0.5,1.5) x U(0, 0.01).
    """
    g = rng(seed)
    blocks = []
    for _ in range(n_blocks):
        blocks.append(dict(qkv=weights(g, 3 * H, H), out=weights(g, H, H),
                           up=weights(g, F, H), down=weights(g, H, F)))
    n_layers = 4 * n_blocks
    alpha = g.uniform(0.5, 1.5, n_layers).astype(np.float32)
    beta = g.uniform(0.0, 0.01, n_layers).astype(np.float32)
    return dict(blocks=blocks, alpha=alpha, beta=beta, noise_seed=int(g.integers(1 << 31)))


def drift_sigma(t: int, n_steps: int) -> float:
    """sigma_t decays linearly from 0.3 (t=0) to 0.01 (t=n_steps-1)."""
    if n_steps <= 1:
        return 0.3
    return 0.3 + (0.01 - 0.3) * t / (n_steps - 1)


def stack_inputs(noise_seed: int, M: int, H: int, n_steps: int):
    """Block-0 inputs of every step: x_0 ~ N(0,1), x_t = x_{t-1} + sigma_t N(0,1)
    (accumulated in float32, stored as bf16 bits per step)."""
    g = rng(noise_seed)
    x = g.standard_normal((M, H), dtype=np.float32)
    xs = [f32_to_bf16_bits(x)]
    for t in range(1, n_steps):
        x = x + np.float32(drift_sigma(t, n_steps)) * g.standard_normal((M, H), dtype=np.float32)
        xs.append(f32_to_bf16_bits(x))
    return xs
