"""Synthetic DiT block and the denoising-step stack with DMPQ and TDC.

Pages: the evaluated models are CogVideoX-2B/5B video DiTs ("Table 1",
"Figure 1" of the thelatestinai.com page); "Figure 2" shows DMPQ choosing
each linear layer's activation bits and TDC skipping whole blocks.  The
trained models are not available; the block below keeps the linear layers
(the only layers the method quantizes) and drops token mixing:

  h1  = LN(x)                         LN without affine, eps 1e-5 (reading)
  qkv = QL(h1; W_qkv);  v = qkv[:, 2H:3H]
  x1  = x + QL(v; W_out)
  h2  = LN(x1)
  u   = GELU_tanh(QL(h2; W_up))
  out = x1 + QL(u; W_down)

QL quantizes its input per the layer's DMPQ flag (NVFP4 -> W4A4, INT8 ->
W4A8) and stores bf16.  Biases are zero.  The stack feeds step t's input to
block 0, chains the blocks, and records the last block's output (reading:
the output is not fed back into the next step's input).

Parity: LN pinned against torch's layer_norm (float64); the block's wiring
pinned by zero weights (the block is then the identity) and by weights
confined to the Q/K rows (the V slice is zero, so x1 = x); the stack's rules
pinned by properties (TDC off == tau_tdc = 0, forced flags == tau = inf, the
alternating skip pattern under max_skip = 1).
"""
from __future__ import annotations

import numpy as np

from . import nvfp4, int8, gemm, gamma, dmpq, tdc
from .codecs import bf16_to_f32, f64_to_bf16

LN_EPS = 1e-5


def layernorm(x_bits, eps: float = LN_EPS):
    x = bf16_to_f32(x_bits).astype(np.float64)
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    return f64_to_bf16((x - mu) / np.sqrt(var + eps))


def quantize_weights(w_f32):
    codes, sf, g, _ = nvfp4.quantize(np.asarray(w_f32, dtype=np.float32))
    return dict(codes=codes, sf=sf, g=g)


def qlinear(h_bits, wq, use_nvfp4: bool, gelu=False, residual=None):
    h = bf16_to_f32(h_bits)
    if use_nvfp4:
        codes, sf, g, _ = nvfp4.quantize(h)
        return gemm.w4a4(codes, sf, g, wq["codes"], wq["sf"], wq["g"], gelu=gelu,
                         residual=residual, out_dtype="bf16")
    q, s, _ = int8.quantize(h)
    return gemm.w4a8(q, s, wq["codes"], wq["sf"], wq["g"], gelu=gelu,
                     residual=residual, out_dtype="bf16")


def block_forward(x_bits, wq_block, flags):
    """flags: 4 uint8 (qkv, out, up, down); 1 = NVFP4."""
    H = x_bits.shape[1]
    h1 = layernorm(x_bits)
    qkv = qlinear(h1, wq_block["qkv"], bool(flags[0]))
    v = np.ascontiguousarray(qkv[:, 2 * H:3 * H])
    x1 = qlinear(v, wq_block["out"], bool(flags[1]), residual=x_bits)
    h2 = layernorm(x1)
    u = qlinear(h2, wq_block["up"], bool(flags[2]), gelu=True)
    return qlinear(u, wq_block["down"], bool(flags[3]), residual=x1)


def run_stack(x_steps, wq_blocks, alpha, beta, tau, tau_tdc, max_skip=1, use_tdc=True,
              forced_flags=None, forced_skips=None, refresh_every=0):
    """Run every step.  Returns dict(outputs, flags[t], skips[t], gammas[t], r2[t]).

    forced_flags (optional) [steps][layers] replaces DMPQ's decisions and
    forced_skips (optional) [steps][blocks] replaces TDC's (teacher forcing
    for parity checks of a free-running device stack).
    """
    nb = len(wq_blocks)
    layer_block = np.repeat(np.arange(nb), 4)
    caches = [tdc.BlockCache() for _ in range(nb)]
    g_prev = np.zeros(nb, dtype=np.float32)
    out_log = dict(outputs=[], flags=[], skips=[], gammas=[], r2=[])
    for t, x in enumerate(x_steps):
        if forced_flags is not None:
            flags = np.asarray(forced_flags[t], dtype=np.uint8)
        else:
            flags = dmpq.assign(g_prev, alpha, beta, layer_block, tau, t)
        g_t = np.zeros(nb, dtype=np.float32)
        skips = np.zeros(nb, dtype=np.uint8)
        h = x
        for l in range(nb):
            c = caches[l]
            if forced_skips is not None:
                skip = bool(forced_skips[t][l])
            else:
                skip = use_tdc and tdc.decide(c, tau_tdc, max_skip, refresh_every, t)
            if skip:
                out = tdc.apply(h, c.delta)
                tdc.after_skip(c)
            else:
                out = block_forward(h, wq_blocks[l], flags[4 * l:4 * l + 4])
            G, dn, r2 = gamma.block_pass(h, out, c.delta, computed=not skip)
            if not skip:
                tdc.after_compute(c, dn, r2)
            g_t[l] = G
            skips[l] = skip
            h = out
        out_log["outputs"].append(h)
        out_log["flags"].append(flags)
        out_log["skips"].append(skips)
        out_log["gammas"].append(g_t)
        out_log["r2"].append(np.array([c.r2 for c in caches], dtype=np.float32))
        g_prev = g_t
    return out_log
