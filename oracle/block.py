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

Fused producers (`fused=True`, an extension, not from the pages): the
three layer inputs whose producer can quantize them in one pass -- h1 and h2
(the LayerNorms) and u (the up-projection's GELU epilogue) -- take NVFP4 by
delayed scaling (nvfp4.quantize_delayed) from a per-block history of their
exact tensor amaxes at the block's previous computed step; INT8 stays exact
(a per-row amax is known to a row-owning producer).  The history is updated
with this step's exact amaxes of h1, h2, u whenever the block is computed,
whatever format each layer took, and left alone when TDC skips the block.
The V slice (the out-projection's input) is quantized as before.

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
F32 = np.float32


def layernorm(x_bits, eps: float = LN_EPS):
    x = bf16_to_f32(x_bits).astype(np.float64)
    mu = x.mean(axis=1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
    return f64_to_bf16((x - mu) / np.sqrt(var + eps))


def quantize_weights(w_f32, chunk_rows=None, keep_dequantized=False):
    """NVFP4 weight: codes, scale bytes, g.  chunk_rows: quantize that many
    rows at a time with the whole matrix's amax (the same result, less
    memory for large matrices).  keep_dequantized: also keep the decoded
    float64 matrix ("deq") for repeated products."""
    w = np.asarray(w_f32, dtype=np.float32)
    if chunk_rows is None:
        codes, sf, g, _ = nvfp4.quantize(w)
    else:
        amax = nvfp4.tensor_amax(w)
        parts = [nvfp4.quantize(w[i:i + chunk_rows], amax) for i in range(0, w.shape[0], chunk_rows)]
        codes = np.concatenate([p[0] for p in parts])
        sf = np.concatenate([p[1] for p in parts])
        g = parts[0][2]
    wq = dict(codes=codes, sf=sf, g=g)
    if keep_dequantized:
        wq["deq"] = nvfp4.dequantize(codes, sf)
    return wq


def qlinear(h_bits, wq, use_nvfp4: bool, gelu=False, residual=None, amax_t=None):
    """amax_t: the NVFP4 tensor amax to quantize with (None: the input's own;
    given when h_bits is a row subset of the layer's whole input)."""
    h = bf16_to_f32(h_bits)
    if use_nvfp4:
        codes, sf, g, _ = nvfp4.quantize(h, amax_t)
        return gemm.w4a4(codes, sf, g, wq["codes"], wq["sf"], wq["g"], gelu=gelu,
                         residual=residual, out_dtype="bf16", w_deq=wq.get("deq"))
    q, s, _ = int8.quantize(h)
    return gemm.w4a8(q, s, wq["codes"], wq["sf"], wq["g"], gelu=gelu,
                     residual=residual, out_dtype="bf16", w_deq=wq.get("deq"))


def block_forward(x_bits, wq_block, flags, amax_hist=None, headroom=2.0, layer_amax=None):
    """flags: 4 uint8 (qkv, out, up, down); 1 = NVFP4.

    amax_hist (fused producers): float32 [3] history of the tensor amaxes of
    h1, h2, u; their NVFP4 layers quantize with headroom * history, and the
    array is overwritten with this call's exact amaxes.
    layer_amax (unfused, optional): the NVFP4 tensor amaxes of the four layer
    inputs (h1, v, h2, u) when x_bits is a row subset of the block input:
    the one quantity of the block that is not computed row by row."""
    H = x_bits.shape[1]
    fused = amax_hist is not None
    used = [F32(F32(headroom) * F32(a)) for a in amax_hist] if fused else [None] * 3
    la = [None] * 4 if layer_amax is None else [F32(a) for a in layer_amax]
    if not fused and layer_amax is not None:
        used = [la[0], la[2], la[3]]
    h1 = layernorm(x_bits)
    qkv = qlinear(h1, wq_block["qkv"], bool(flags[0]), amax_t=used[0])
    v = np.ascontiguousarray(qkv[:, 2 * H:3 * H])
    x1 = qlinear(v, wq_block["out"], bool(flags[1]), residual=x_bits, amax_t=la[1])
    h2 = layernorm(x1)
    u = qlinear(h2, wq_block["up"], bool(flags[2]), gelu=True, amax_t=used[1])
    out = qlinear(u, wq_block["down"], bool(flags[3]), residual=x1, amax_t=used[2])
    if fused:
        for i, t in enumerate((h1, h2, u)):
            amax_hist[i] = nvfp4.tensor_amax(bf16_to_f32(t))
    return out


def run_stack(x_steps, wq_blocks, alpha, beta, tau, tau_tdc, max_skip=1, use_tdc=True,
              forced_flags=None, forced_skips=None, refresh_every=0, fused=False, headroom=2.0, tdc_cache="bf16"):
    """Run every step.  Returns dict(outputs, flags[t], skips[t], gammas[t], r2[t]).

    fused: fused producers with delayed NVFP4 scaling (module header); every
    block's amax history starts at zero.  tdc_cache: "bf16", or "mx" for the
    compressed update cache of oracle.mxcache (an extension).

    forced_flags (optional) [steps][layers] replaces DMPQ's decisions and
    forced_skips (optional) [steps][blocks] replaces TDC's (teacher forcing
    for parity checks of a free-running device stack).
    """
    nb = len(wq_blocks)
    layer_block = np.repeat(np.arange(nb), 4)
    caches = [tdc.BlockCache() for _ in range(nb)]
    hist = [np.zeros(3, dtype=F32) if fused else None for _ in range(nb)]
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
                out = block_forward(h, wq_blocks[l], flags[4 * l:4 * l + 4], hist[l], headroom)
            G, dn, r2 = gamma.block_pass(h, out, c.delta, computed=not skip, cache=tdc_cache)
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
        if fused:
            out_log.setdefault("amax_hist", []).append(np.stack(hist))
        g_prev = g_t
    return out_log
