"""Synthetic DiT block stack driven through the sixbit C ABI, with DMPQ and TDC.

Block (the linear layers of a video-DiT block; token mixing omitted):
    h1 = LN(x); qkv = QL(h1); x1 = x + QL(qkv[:, 2H:3H]); h2 = LN(x1);
    u = GELU(QL(h2)); out = x1 + QL(u)
QL quantizes its input to NVFP4 (W4A4) or INT8 (W4A8) as the layer's DMPQ
flag says.  6Bit-Diffusion (thelatestinai.com page, Figure 2): DMPQ picks
each layer's activation bits from the block's Gamma at the previous step;
TDC skips a block whose update barely changed and reuses in + Delta.

Fused producers (fused=True; an extension, not from the pages): the
LayerNorms quantize their own outputs (INT8 exactly per row, NVFP4 by
delayed scaling from a per-layer amax history) and the up-projection's GELU
epilogue writes the down layer's NVFP4 input directly, so h1, h2 and (for an
NVFP4 down layer) u never round-trip through HBM as bf16; the quantizer
passes of those layers disappear.  The V slice keeps its own quantizer.

Every decision stays on the device.  At the start of a step DMPQ writes one
gate byte per (layer, format); the TDC kernel of a block clears the block's
gates when it skips it; every kernel of the block reads its gate (`pred`)
and exits at once when it is 0.  One step is captured once as a CUDA graph
and replayed; only the block-0 input and the step counter are written
between replays.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (amax_hist_value, amax_history, block_gamma, dmpq_assign, layernorm, layernorm_quant, mxcache,
               qlinear_qout, qlinear_w4a4,
               qlinear_w4a8, quantize_act_int8, quantize_act_nvfp4, quantize_weight_nvfp4, sf_bytes,
               tdc_decide_and_apply)

LN_EPS = 1e-5
LAYERS = ("qkv", "out", "up", "down")


class DiTStack:
    """n_blocks blocks of hidden size H and FFN size F over M tokens.

    weights: list (per block) of dicts qkv [3H,H], out [H,H], up [F,H], down [H,F]
    (float32 numpy or torch); alpha, beta: per-layer predictor lines (4 per
    block, layer order qkv, out, up, down); tau: DMPQ threshold; tau_tdc,
    max_skip: TDC rule (max_skip = 0 disables skipping); refresh_every: PDR
    periodic refresh (every k-th step is computed; 0 = off); fused: quantizing
    producers with delayed NVFP4 scaling (headroom: its power-of-two margin);
    tdc_cache: "bf16" (one bf16 update per block) or "mx" (the compressed
    cache: E4M3 codes with a power-of-two scale per 32 elements).
    """

    def __init__(self, weights, alpha, beta, M: int, H: int, F: int, tau: float, tau_tdc: float = 0.05,
                 max_skip: int = 1, device=None, refresh_every: int = 0, fused: bool = False,
                 headroom: float = 2.0, tdc_cache: str = "bf16"):
        self.dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        dev = self.dev
        self.nb, self.M, self.H, self.F = len(weights), M, H, F
        self.tau, self.tau_tdc, self.max_skip = float(tau), float(tau_tdc), int(max_skip)
        self.refresh_every = int(refresh_every)
        self.fused, self.headroom = bool(fused), float(headroom)
        nl = 4 * self.nb
        to_t = lambda a: torch.as_tensor(np.asarray(a, np.float32)).to(dev)
        self.alpha, self.beta = to_t(alpha), to_t(beta)
        self.layer_block = torch.arange(self.nb, dtype=torch.int32, device=dev).repeat_interleave(4)
        self.wq = []
        for b in weights:
            self.wq.append({k: quantize_weight_nvfp4(torch.as_tensor(b[k]).to(dev, torch.float32).contiguous())
                            for k in LAYERS})
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.x_in = torch.zeros((M, H), **bf)
        self.buf = [torch.zeros((M, H), **bf), torch.zeros((M, H), **bf)]
        self.h1 = torch.empty((M, H), **bf)
        self.qkv = torch.empty((M, 3 * H), **bf)
        self.x1 = torch.empty((M, H), **bf)
        self.h2 = torch.empty((M, H), **bf)
        self.u = torch.empty((M, F), **bf)
        kmax = max(H, F)
        self.codes = torch.empty(M * kmax // 2, dtype=torch.uint8, device=dev)
        self.sf = torch.empty(sf_bytes(M, kmax), dtype=torch.uint8, device=dev)
        self.g = torch.empty(1, dtype=torch.float32, device=dev)
        self.planes = torch.empty(3 * M * kmax // 2, dtype=torch.uint8, device=dev)
        self.rs = torch.empty(M, dtype=torch.float32, device=dev)
        self.amax = torch.empty(1, dtype=torch.float32, device=dev)
        self.row_amax = torch.empty(M, dtype=torch.float32, device=dev)
        # fused producers: the down layer's NVFP4 input (written by the up
        # epilogue) and one delayed-scaling history per producer (LN1, LN2, up)
        self.hist = amax_history(3 * self.nb, dev)
        # unfused: the up-projection's exact |u| amax, a side output of its GEMM
        # that lets the down layer's NVFP4 quantizer skip its amax pass
        self.u_amax = amax_history(1, dev)[0]
        if self.fused:
            self.codes_u = torch.empty((M, F // 2), dtype=torch.uint8, device=dev)
            self.sf_u = torch.empty(sf_bytes(M, F), dtype=torch.uint8, device=dev)
            self.g_u = torch.empty(1, dtype=torch.float32, device=dev)
        # decisions and TDC cache
        self.step_dev = torch.zeros(1, dtype=torch.int32, device=dev)
        self.use_nvfp4 = torch.zeros(nl, dtype=torch.uint8, device=dev)
        self.gates = torch.zeros((nl, 2), dtype=torch.uint8, device=dev)
        self.gamma = torch.zeros(self.nb, dtype=torch.float32, device=dev)
        if tdc_cache not in ("bf16", "mx"):
            raise ValueError("tdc_cache is 'bf16' or 'mx'")
        self.tdc_cache = tdc_cache
        self.delta = [torch.zeros((M, H), **bf) if tdc_cache == "bf16" else mxcache(M * H, dev)
                      for _ in range(self.nb)]
        self.r2 = torch.full((self.nb,), float("inf"), dtype=torch.float32, device=dev)
        self.state = torch.zeros((self.nb, 2), dtype=torch.int32, device=dev)
        self.cflag = torch.ones(self.nb, dtype=torch.uint8, device=dev)
        self.graph = None
        self.out = self.buf[(self.nb - 1) % 2]

    def set_tdc_cache(self, fmt: str):
        """Switch the update cache format ("bf16" / "mx"); clears the caches and
        drops the captured graph."""
        if fmt not in ("bf16", "mx"):
            raise ValueError("tdc_cache is 'bf16' or 'mx'")
        if fmt != self.tdc_cache:
            M, H = self.M, self.H
            self.delta = [torch.zeros((M, H), dtype=torch.bfloat16, device=self.dev) if fmt == "bf16"
                          else mxcache(M * H, self.dev) for _ in range(self.nb)]
            self.tdc_cache = fmt
        self.graph = None

    # ------------------------------------------------------------ one step
    def _ql(self, x, wq, gate_nv, gate_i8, out, amax_in=None, row_amax_in=None, residual=None, gelu=False,
            amax_side=None):
        """Quantize x as the gates say and run the layer.  amax_side: a history
        row that receives max |out| (the GEMM's exact amax side output)."""
        M, K = x.shape
        codes = self.codes[:M * K // 2].view(M, K // 2)
        sf = self.sf[:sf_bytes(M, K)]
        planes = self.planes[:3 * M * K // 2].view(3, M, K // 2)
        quantize_act_nvfp4(x, amax_in=amax_in, pred=gate_nv, out=(codes, sf, self.g))
        if amax_side is None:
            qlinear_w4a4(codes, sf, self.g, *wq, residual=residual, gelu=gelu, out=out, pred=gate_nv)
        else:
            qlinear_qout("w4a4", codes, *wq, None, None, None, amax_side, a_sf=sf, g_a=self.g, gelu=gelu, y=out,
                         pred=gate_nv)
        quantize_act_int8(x, row_amax=row_amax_in, want_q=False, pred=gate_i8, out=(None, planes, self.rs))
        if amax_side is None:
            qlinear_w4a8(planes, self.rs, *wq, residual=residual, gelu=gelu, out=out, pred=gate_i8)
        else:
            qlinear_qout("w4a8", planes, *wq, None, None, None, amax_side, row_scale=self.rs, gelu=gelu, y=out,
                         pred=gate_i8)

    def _ln_q(self, x, i, l, gates, c, keep_bf16):
        """Fused LayerNorm feeding layer i of block l: NVFP4 / INT8 as its gates say."""
        H, M = self.H, self.M
        y = self.h1 if i == 0 else self.h2
        layernorm_quant(x, LN_EPS, y=y if keep_bf16 else None,
                        nvfp4=(self.codes[:M * H // 2].view(M, H // 2), self.sf[:sf_bytes(M, H)], self.g),
                        amax_hist=self.hist[3 * l + (0 if i == 0 else 1)], headroom=self.headroom,
                        nv_pred=gates[i, 0:1],
                        int8=(self.planes[:3 * M * H // 2].view(3, M, H // 2), self.rs), i8_pred=gates[i, 1:2], pred=c)
        return y

    def _ql_from_ln(self, wq, gates, i, out, gelu=False):
        """Layer i's GEMMs on the operands a fused LayerNorm left in the shared buffers."""
        H, M = self.H, self.M
        codes, sf = self.codes[:M * H // 2].view(M, H // 2), self.sf[:sf_bytes(M, H)]
        planes = self.planes[:3 * M * H // 2].view(3, M, H // 2)
        qlinear_w4a4(codes, sf, self.g, *wq, gelu=gelu, out=out, pred=gates[i, 0:1])
        qlinear_w4a8(planes, self.rs, *wq, gelu=gelu, out=out, pred=gates[i, 1:2])

    def _up_down_fused(self, l, gates, out):
        """Up-projection whose GELU epilogue emits the down layer's NVFP4 input
        (or bf16 u for an INT8 down layer), then the down-projection."""
        H, M, F = self.H, self.M, self.F
        codes, sf = self.codes[:M * H // 2].view(M, H // 2), self.sf[:sf_bytes(M, H)]
        planes = self.planes[:3 * M * H // 2].view(3, M, H // 2)
        wu, wd = self.wq[l]["up"], self.wq[l]["down"]
        qo = dict(q_codes=self.codes_u, q_sf=self.sf_u, q_g=self.g_u, amax_hist=self.hist[3 * l + 2],
                  headroom=self.headroom, gelu=True, y=self.u, q_pred=gates[3, 0:1])
        qlinear_qout("w4a4", codes, *wu, a_sf=sf, g_a=self.g, pred=gates[2, 0:1], **qo)
        qlinear_qout("w4a8", planes, *wu, row_scale=self.rs, pred=gates[2, 1:2], **qo)
        qlinear_w4a4(self.codes_u, self.sf_u, self.g_u, *wd, residual=self.x1, out=out, pred=gates[3, 0:1])
        planes_u = self.planes[:3 * M * F // 2].view(3, M, F // 2)
        quantize_act_int8(self.u, want_q=False, pred=gates[3, 1:2], out=(None, planes_u, self.rs))
        qlinear_w4a8(planes_u, self.rs, *wd, residual=self.x1, out=out, pred=gates[3, 1:2])

    def enqueue_step(self, hook=None, block_hook=None):
        """Enqueue one denoising step on the current stream (graph-capturable).
        hook (eager calibration runs only): called as hook(block, layer_index,
        x) with each linear layer's bf16 input before the layer runs.
        block_hook (eager runs only): called as block_hook(block, x_in, x_out)
        just before the block's Gamma pass, when the update cache still holds
        the previous update; work it enqueues on the stream sees the block's
        input and output."""
        if self.fused:
            if hook is not None:
                raise ValueError("calibration hooks need the unfused stack (fused=False)")
            return self._enqueue_fused(block_hook)
        H = self.H
        call = (lambda l, i, x: hook(l, i, x)) if hook is not None else (lambda l, i, x: None)
        dmpq_assign(self.gamma, self.alpha, self.beta, self.layer_block, self.tau, self.step_dev,
                    use_nvfp4=self.use_nvfp4, gates=self.gates)
        h = self.x_in
        for l in range(self.nb):
            out = self.buf[l % 2]
            gates = self.gates[4 * l:4 * l + 4]
            c = self.cflag[l:l + 1]
            tdc_decide_and_apply(h, self.delta[l], self.r2[l:l + 1], self.tau_tdc, self.max_skip, self.state[l],
                                 c, out, gates=gates, refresh_every=self.refresh_every, step=self.step_dev)
            g = lambda i, f: gates[i, f:f + 1]
            layernorm(h, LN_EPS, out=self.h1, amax_out=self.amax, row_amax_out=self.row_amax, pred=c)
            call(l, 0, self.h1)
            self._ql(self.h1, self.wq[l]["qkv"], g(0, 0), g(0, 1), self.qkv, amax_in=self.amax,
                     row_amax_in=self.row_amax)
            v = self.qkv[:, 2 * H:3 * H]
            call(l, 1, v)
            self._ql(v, self.wq[l]["out"], g(1, 0), g(1, 1), self.x1, residual=h)
            layernorm(self.x1, LN_EPS, out=self.h2, amax_out=self.amax, row_amax_out=self.row_amax, pred=c)
            call(l, 2, self.h2)
            self._ql(self.h2, self.wq[l]["up"], g(2, 0), g(2, 1), self.u, amax_in=self.amax,
                     row_amax_in=self.row_amax, gelu=True, amax_side=self.u_amax)
            call(l, 3, self.u)
            self._ql(self.u, self.wq[l]["down"], g(3, 0), g(3, 1), out, residual=self.x1,
                     amax_in=amax_hist_value(self.u_amax))
            if block_hook is not None:
                block_hook(l, h, out)
            block_gamma(h, out, delta=self.delta[l], gamma_out=self.gamma[l:l + 1], r2_out=self.r2[l:l + 1],
                        tdc_state=self.state[l], computed=c)
            h = out
        self.out = h

    def _enqueue_fused(self, block_hook=None):
        H = self.H
        dmpq_assign(self.gamma, self.alpha, self.beta, self.layer_block, self.tau, self.step_dev,
                    use_nvfp4=self.use_nvfp4, gates=self.gates)
        h = self.x_in
        for l in range(self.nb):
            out = self.buf[l % 2]
            gates = self.gates[4 * l:4 * l + 4]
            c = self.cflag[l:l + 1]
            tdc_decide_and_apply(h, self.delta[l], self.r2[l:l + 1], self.tau_tdc, self.max_skip, self.state[l],
                                 c, out, gates=gates, refresh_every=self.refresh_every, step=self.step_dev)
            g = lambda i, f: gates[i, f:f + 1]
            self._ln_q(h, 0, l, gates, c, keep_bf16=False)
            self._ql_from_ln(self.wq[l]["qkv"], gates, 0, self.qkv)
            v = self.qkv[:, 2 * H:3 * H]
            self._ql(v, self.wq[l]["out"], g(1, 0), g(1, 1), self.x1, residual=h)
            self._ln_q(self.x1, 2, l, gates, c, keep_bf16=False)
            self._up_down_fused(l, gates, out)
            if block_hook is not None:
                block_hook(l, h, out)
            block_gamma(h, out, delta=self.delta[l], gamma_out=self.gamma[l:l + 1], r2_out=self.r2[l:l + 1],
                        tdc_state=self.state[l], computed=c)
            h = out
        self.out = h

    def capture(self):
        """Warm up once (kernel attributes, scratch) and capture one step as a CUDA graph."""
        snap = self._snapshot()
        self.enqueue_step()
        torch.cuda.synchronize()
        self._restore(snap)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.enqueue_step()
        torch.cuda.synchronize()

    def _state_tensors(self):
        return (self.gamma, self.r2, self.state, self.cflag, self.use_nvfp4, self.gates, self.hist)

    def _snapshot(self):
        return [t.clone() for t in self._state_tensors()] + [d.clone() for d in self.delta]

    def _restore(self, snap):
        n = len(self._state_tensors())
        for t, s in zip(self._state_tensors(), snap[:n]):
            t.copy_(s)
        for d, s in zip(self.delta, snap[n:]):
            d.copy_(s)

    def reset(self):
        self.gamma.zero_()
        self.r2.fill_(float("inf"))
        self.state.zero_()
        self.cflag.fill_(1)
        self.use_nvfp4.zero_()
        self.gates.zero_()
        self.hist.zero_()
        for d in self.delta:
            d.zero_()

    def run(self, xs, record=False):
        """Run every step with block-0 inputs xs (list of bf16 [M,H] device tensors).

        Returns the last block's output of every step (clones) and, with
        record=True, per-step decisions: flags [steps, layers], skips
        [steps, blocks], gamma, r2 and the TDC counters after the step.
        """
        if self.graph is None:
            self.capture()
        outs, log = [], dict(flags=[], skips=[], gamma=[], r2=[], state=[])
        for t, x in enumerate(xs):
            self.x_in.copy_(x)
            self.step_dev.fill_(t)
            self.graph.replay()
            outs.append(self.out.clone())
            if record:
                log["flags"].append(self.use_nvfp4.clone())
                log["skips"].append(1 - self.cflag)
                log["gamma"].append(self.gamma.clone())
                log["r2"].append(self.r2.clone())
                log["state"].append(self.state.clone())
        return outs, log
