"""Benchmark of the 6Bit-Diffusion hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload 2b|5b]

One step = one pass of the whole hot path over one batch of synthetic input
shaped like the 2B-class video-DiT GEMM set (M = 17776 tokens):
for each linear layer (QKV 1920->5760, out-proj 1920->1920 + residual,
FFN-up 1920->7680 + GELU, FFN-down 7680->1920 + residual)
    NVFP4: tensor amax -> quantize -> W4A4 GEMM (bf16 out)
    INT8:  per-token quantize (digit planes) -> W4A8 GEMM (bf16 out)
then the block Gamma/Delta/r2 pass over a [M, 1920] block input/output,
DMPQ assignment of the block's 4 layers, and the TDC decision.
Weights are quantized once (offline) before timing.

value = quantized-linear TFLOP/s = sum over the 8 GEMMs of 2MNK / step time
(inputs already in HBM).  The working set of a step (~1.5 GB) is larger than
the 129 MB L2, so no explicit flush is done between steps.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the reference arm); other ranks exit at once.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic  # noqa: E402

METRIC = "quantized-linear TFLOPS (NVFP4, INT8) + DiT blocks/s w/ DMPQ+TDC; % roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense FP4 : BF16 tensor ratio on GB300


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK, "fallback"


def workload_layers(name: str):
    return synthetic.GEMM_SHAPES["2B" if name == "2b" else "5B"]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The largest x over the ranks of the initialised process group (the
    job's timed region ends when its slowest rank ends); x itself when ws == 1.
    device: where the reduction tensor lives (the GPU for NCCL, None = CPU for gloo)."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ws: int, elapsed_max: float) -> float:
    """Whole-job throughput: every rank's units (weak scaling: the same work
    per rank) over the slowest rank's time."""
    return units_per_rank * ws / elapsed_max


def gemm_roofline(mode: str, M: int, N: int, K: int, residual: bool, seconds: float,
                  fp4_peak_tflops: float, hbm_gbs: float) -> dict:
    """Roofline of one quantized-linear launch against the method's own work.

    FLOPs: 2MNK.  Algorithmic bytes: the activation operand in the method's
    format (W4A4: E2M1 codes + E4M3 block scales; W4A8: int8 codes + fp32 row
    scales), the NVFP4 weight (codes + scales), the bf16 output and, with a
    residual, its bf16 read.  Ceiling: min(dense FP4 tensor peak, HBM x AI).
    W4A8 runs on the FP4 pipe as three exact digit-plane MMAs per product,
    so its `fp4_pipe_frac` (3 x its FLOP rate / FP4 peak) is how busy that
    pipe is, and `design_ceiling` = FP4 peak / 3 is the most this design can
    reach; `bytes_moved` counts the digit planes (1.5 B/element) it streams
    instead of the 1-byte codes."""
    flops = 2.0 * M * N * K
    w_bytes = N * K / 2 + N * K / 16
    y_bytes = 2.0 * M * N * (2 if residual else 1)
    if mode == "w4a8":
        a_bytes, a_moved = M * K + 4 * M, 1.5 * M * K + 4 * M
    else:
        a_bytes = a_moved = M * K / 2 + M * K / 16
    nbytes = a_bytes + w_bytes + y_bytes
    ai = flops / nbytes
    hbm = hbm_gbs * ai / 1e3                    # GB/s x FLOP/B -> TFLOP/s
    ceiling = min(fp4_peak_tflops, hbm)
    achieved = flops / seconds / 1e12
    r = {"ms": seconds * 1e3, "TFLOP/s": achieved, "bytes": nbytes, "bytes_moved": a_moved + w_bytes + y_bytes,
         "AI": ai, "bound": "tensor" if fp4_peak_tflops <= hbm else "hbm", "ceiling": ceiling,
         "frac_ceiling": achieved / ceiling, "frac_fp4_peak": achieved / fp4_peak_tflops}
    if mode == "w4a8":
        r["fp4_pipe_frac"] = 3.0 * achieved / fp4_peak_tflops
        r["design_ceiling"] = fp4_peak_tflops / 3.0
    return r


def quant_bytes(kind: str, M: int, K: int) -> float:
    """Algorithmic bytes of an activation quantizer over [M, K]: read bf16 x
    once, write the method's format (NVFP4: 0.5 B codes + 1/16 B E4M3 scales
    per element; INT8: 1 B codes per element + a 4-byte row scale)."""
    if kind == "nvfp4":
        return (2 + 0.5 + 1 / 16) * M * K
    return 3.0 * M * K + 4.0 * M


def stack_ideal_seconds(M: int, H: int, F: int, nv_computed, i8_computed, computed, skipped,
                        fp4_peak_tflops: float, hbm_gbs: float) -> float:
    """Sum of per-kernel roofline times of a DiT stack run (the time-weighted
    bound): for every computed block evaluation two LayerNorms (bf16 in and
    out, with their amax side outputs), per layer the quantizer of its format
    (NVFP4: the V slice's own amax pass, then 2.5625 B/element; INT8:
    3 B/element) and its GEMM at min(FP4 peak, HBM x AI) (W4A8 at a third of
    the FP4 peak: its three digit-plane MMAs), the Gamma/Delta pass (8 B per
    element); for a skipped block the TDC reuse (6 B/element) and the Gamma
    pass.  nv_computed / i8_computed: per layer kind (qkv, out, up, down) the
    number of computed evaluations in that format; computed / skipped: block
    evaluation counts."""
    shapes = {"qkv": (H, 3 * H, False), "out": (H, H, True), "up": (H, F, False), "down": (F, H, True)}
    t = 0.0
    for k, (K, N, res) in shapes.items():
        for mode, count in (("w4a4", nv_computed[k]), ("w4a8", i8_computed[k])):
            if not count:
                continue
            g = gemm_roofline(mode, M, N, K, res, 1.0, fp4_peak_tflops, hbm_gbs)
            tensor = fp4_peak_tflops / (3.0 if mode == "w4a8" else 1.0)
            gemm_s = 2.0 * M * N * K / (min(tensor, g["ceiling"]) * 1e12)
            qb = quant_bytes("nvfp4" if mode == "w4a4" else "int8", M, K)
            if mode == "w4a4" and k == "out":
                qb += 2.0 * M * K                  # the V slice's tensor amax pass (no producer supplies it)
            t += count * (gemm_s + qb / (hbm_gbs * 1e9))
    ln = 2 * (4.0 * M * H)                        # two LayerNorms, bf16 in and out
    t += computed * (ln + 8.0 * M * H) / (hbm_gbs * 1e9)
    t += skipped * (6.0 * M * H + 8.0 * M * H) / (hbm_gbs * 1e9)
    return t


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", gpu_id], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.tmp.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.tmp.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- ncu traffic
def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_fp4.cu", "common.cuh"):
        with open(os.path.join(ROOT, "nvfp4_int8_mixed_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none or the GEMM source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = None
    vals = {}
    for line in open(path):
        line = line.strip()
        if line.startswith("source_sha256_16:"):
            src = line.split(":", 1)[1].strip()
        elif line and not line.startswith("#") and "=" in line:
            k, v = line.split("=", 1)
            try:
                vals[k.strip()] = float(v)
            except ValueError:
                pass
    if src != kernel_source_hash():
        return None
    return vals.get(kernel)


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(layers, rows_per_layer: int, cols_per_layer: int, seed: int, M: int, prep=None):
    """Prepare (untimed) oracle inputs for a sample: row/column subsets of
    every layer, weights quantized by the oracle itself."""
    from oracle import codecs, nvfp4
    if prep is not None:
        return prep
    out = []
    rng = np.random.default_rng(seed)
    for li, (name, K, N, gelu, res) in enumerate(layers):
        lay = synthetic.gemm_layer(1, M, K, N, res)
        af = codecs.bf16_to_f32(lay["a"])
        amax_t = np.float32(np.max(np.abs(af)))
        rows = rng.choice(M, rows_per_layer, replace=False)
        cols = rng.choice(N, cols_per_layer, replace=False)
        wc, wsf, gw, _ = nvfp4.quantize(lay["w"][cols])
        out.append(dict(a=af[rows], amax=amax_t, wc=wc, wsf=wsf, gw=gw, gelu=gelu,
                        res=None if lay["residual"] is None else lay["residual"][rows][:, cols], K=K))
    g = synthetic.gamma_pair(7, 64, 1920)
    return dict(layers=out, gamma=g)


def oracle_step(prep):
    """One bounded oracle pass: quantize + both GEMMs per layer sample, Gamma,
    DMPQ, TDC decision.  Returns the algorithmic FLOPs it covered."""
    from oracle import dmpq, gamma, gemm, int8, nvfp4, tdc
    flops = 0
    for L in prep["layers"]:
        c, s, g, _ = nvfp4.quantize(L["a"], L["amax"])
        gemm.w4a4(c, s, g, L["wc"], L["wsf"], L["gw"], gelu=L["gelu"], residual=L["res"], out_dtype="bf16")
        q, sc, _ = int8.quantize(L["a"])
        gemm.w4a8(q, sc, L["wc"], L["wsf"], L["gw"], gelu=L["gelu"], residual=L["res"], out_dtype="bf16")
        flops += 2 * 2 * L["a"].shape[0] * L["wc"].shape[0] * L["K"]
    p = prep["gamma"]
    G, dn, r2 = gamma.block_pass(p["xin"], p["xout"], p["delta_prev"])
    dmpq.assign(np.array([G]), np.ones(4, np.float32), np.zeros(4, np.float32), np.zeros(4, np.int64), 0.1, 1)
    tdc.decide(tdc.BlockCache(fresh_count=2, r2=r2), 0.05, 1)
    return flops


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max([i.get("num_threads", 1) for i in info] or [1])
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def time_oracle(layers, M, rows, cols, steps=1, warmup=0, seed=0):
    prep = oracle_sample(layers, rows, cols, seed, M)
    for _ in range(warmup):
        oracle_step(prep)
    t0 = time.perf_counter()
    flops = 0
    for _ in range(steps):
        flops += oracle_step(prep)
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, flops


# ---------------------------------------------------------------- reference arm
def workload_config(workload: str, M: int, layers, ws: int) -> dict:
    """The `config` of the JSON line, the same for both arms."""
    return {"workload": f"{workload.upper()}-class video-DiT GEMM set, M={M} tokens, "
                        "4 linears x (NVFP4+W4A4, INT8+W4A8) + Gamma/DMPQ/TDC",
            "shapes": [[name, M, K, N] for name, K, N, _, _ in layers], "l2": "inputs larger than L2",
            "parallelism": f"replicas x{ws}"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    layers = workload_layers(args.workload)
    M = synthetic.M_2B if args.workload == "2b" else synthetic.M_2B
    rows, cols = 8, 128
    prep = oracle_sample(layers, rows, cols, 0, M)
    for _ in range(args.warmup):
        oracle_step(prep)
    t0 = time.perf_counter()
    flops = sum(oracle_step(prep) for _ in range(args.steps))
    dt = time.perf_counter() - t0
    v = flops / dt / 1e12
    sample = (f"per step: {rows} random rows x {cols} random output columns of each of the 4 layers, "
              f"NVFP4+W4A4 and INT8+W4A8, plus Gamma/DMPQ/TDC on a 64x1920 block pair")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, M, layers, ws),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- DiT stack
STACKS = {
    "2b": dict(n_blocks=30, M=synthetic.M_2B, H=1920, F=7680, steps=50, seed=3, calib_steps=10),
    "5b": dict(n_blocks=42, M=2 * synthetic.M_2B, H=3072, F=12288, steps=50, seed=4),   # CFG batch 2
}


def time_producers(sb, L, dev, gpair, reps=24):
    """Quantizing producers and the compressed-cache Gamma pass at the 2B
    shapes: the LayerNorm over the FFN input (M x 1920) with each output, the
    FFN up-projection (GELU) whose epilogue emits the down layer's NVFP4
    input, and the Gamma / Delta / r2 pass with the bf16 and the compressed
    update cache.  Each is `reps` launches captured as one CUDA graph and
    replayed between CUDA events (median of 5 replays, divided by `reps`);
    the LayerNorm and Gamma launches rotate over input copies whose total
    exceeds L2, so their inputs come from HBM and no flush leaves dirty lines
    to be written back during a timed launch."""
    import torch
    x = L[0]["x"]
    M, H = x.shape
    up = next(l for l in L if l["name"] == "ffn_up")
    N = up["N"]
    u8 = dict(dtype=torch.uint8, device=dev)
    codes, sf, g = torch.empty((M, H // 2), **u8), torch.empty(sb.sf_bytes(M, H), **u8), torch.empty(1, device=dev)
    planes, rs = torch.empty((3, M, H // 2), **u8), torch.empty(M, device=dev)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    qc, qsf, qg = torch.empty((M, N // 2), **u8), torch.empty(sb.sf_bytes(M, N), **u8), torch.empty(1, device=dev)
    hist = sb.amax_history(2, dev)
    elt = M * H
    nx = max(2, -(-(300 << 20) // (elt * 2)))            # LayerNorm inputs: > 300 MB in all
    xs = [x] + [x.clone() for _ in range(nx - 1)]
    # Gamma: two (input, output, update cache) sets, 2 x 205 MB
    gsets = [(gpair[0], gpair[1], torch.zeros((M, H), dtype=torch.bfloat16, device=dev), sb.mxcache(elt, dev)),
             (gpair[0].clone(), gpair[1].clone(), torch.zeros((M, H), dtype=torch.bfloat16, device=dev),
              sb.mxcache(elt, dev))]
    st = torch.tensor([1, 0], dtype=torch.int32, device=dev)
    gr = torch.empty(2, dtype=torch.float32, device=dev)

    def gamma_call(i, mx):
        # st[0] >= 1 (one previous update) stays so: each computed pass adds one
        xin, xout, dc, mc = gsets[i % 2]
        sb.block_gamma(xin, xout, delta=mc if mx else dc, gamma_out=gr[0:1], r2_out=gr[1:2], tdc_state=st)

    X = lambda i: xs[i % nx]
    cases = {
        "gamma_delta_bf16_cache": (lambda i: gamma_call(i, False), 8 * elt),
        "gamma_delta_mx_cache": (lambda i: gamma_call(i, True), 4 * elt + 2 * int(sb.lib().sixbit_mxcache_bytes(elt))),
        "layernorm_bf16": (lambda i: sb.layernorm(X(i), out=y), 4 * elt),
        "layernorm_nvfp4": (lambda i: sb.layernorm_quant(X(i), nvfp4=(codes, sf, g), amax_hist=hist[0]), 2.5625 * elt),
        "layernorm_int8": (lambda i: sb.layernorm_quant(X(i), int8=(planes, rs)), quant_bytes("int8", M, H)),
        "layernorm_bf16_nvfp4": (lambda i: sb.layernorm_quant(X(i), y=y, nvfp4=(codes, sf, g), amax_hist=hist[0]),
                                 4.5625 * elt),
        "qout_w4a4[ffn_up]": (lambda i: sb.qlinear_qout("w4a4", up["codes"], up["wc"], up["wsf"], up["gw"], qc, qsf, qg,
                                                         hist[1], a_sf=up["sf"], g_a=up["ga"], gelu=True, y=up["y4"]),
                              None),
        "qout_w4a8[ffn_up]": (lambda i: sb.qlinear_qout("w4a8", up["planes"], up["wc"], up["wsf"], up["gw"], qc, qsf, qg,
                                                         hist[1], row_scale=up["s"], gelu=True, y=up["y4"]), None),
    }
    peak = float(load_peaks()[0]["hbm_gbs"])
    stream = torch.cuda.current_stream()
    out = {}
    for name, (fn, nbytes) in cases.items():
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(reps):
                fn(i)
        graph.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3 / reps)
        sb.get_error()
        del graph
        t = float(np.median(ts))
        if nbytes is None:
            out[name] = {"us": t * 1e6, "TFLOP/s": 2 * M * N * up["K"] / t / 1e12}
        else:
            out[name] = {"us": t * 1e6, "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peak}
    del xs, gsets
    return out


def time_oracle_block(weight_block, x_bits, M: int, row_counts=(128, 512), seed=0):
    """CPU baseline of the stack metric: the oracle's block_forward on one
    block at two row counts (random rows of the block input), timed on the
    host cores; the time is fitted as fixed + per-row cost and extrapolated
    to M rows.  Layer formats: qkv, up NVFP4; out, down INT8."""
    from oracle import block as o_block
    wq = {k: o_block.quantize_weights(np.asarray(v, np.float32)) for k, v in weight_block.items()}
    rng = np.random.default_rng(seed)
    flags = np.array([1, 0, 1, 0], np.uint8)
    ts = []
    for r in row_counts:
        rows = np.sort(rng.choice(x_bits.shape[0], r, replace=False))
        t0 = time.perf_counter()
        o_block.block_forward(x_bits[rows], wq, flags)
        ts.append(time.perf_counter() - t0)
    b = (ts[1] - ts[0]) / (row_counts[1] - row_counts[0])
    a = max(ts[0] - b * row_counts[0], 0.0)
    t_full = a + b * M
    return {"blocks_per_s": 1.0 / t_full, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"oracle block_forward of one block at {row_counts[0]} and {row_counts[1]} random rows "
                      f"({ts[0]:.1f} s, {ts[1]:.1f} s); blocks/s extrapolated linearly in rows to M={M}"}


def bf16_stack_context(weights, xs, H):
    """The same block stack in plain bf16 torch ops (cuBLAS GEMMs), one CUDA
    graph per step: the unquantized "original" the pages compare against.
    Context only; none of the library's kernels run here."""
    import torch
    import torch.nn.functional as Fn
    w = [{k: b[k].to(torch.bfloat16) for k in ("qkv", "out", "up", "down")} for b in weights]
    x_in = torch.empty_like(xs[0])

    def step():
        x = x_in
        for b in w:
            h1 = Fn.layer_norm(x, (H,), eps=1e-5)
            v = (h1 @ b["qkv"].t())[:, 2 * H:]
            x1 = x + v @ b["out"].t()
            u = Fn.gelu(Fn.layer_norm(x1, (H,), eps=1e-5) @ b["up"].t(), approximate="tanh")
            x = x1 + u @ b["down"].t()
        return x

    x_in.copy_(xs[0])
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for t in range(3):
        x_in.copy_(xs[t])
        g.replay()
    torch.cuda.synchronize()
    e0.record()
    for x in xs:
        x_in.copy_(x)
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3
    del g, w
    torch.cuda.empty_cache()
    return {"blocks_per_s": len(weights) * len(xs) / sec, "ms_per_step": sec / len(xs) * 1e3}


def run_stack_bench(name: str, dev, cpu_oracle: bool = False, modes=None):
    """Blocks/s of the synthetic DiT stack with DMPQ+TDC and with DMPQ only.

    Weights N(0, 0.02) and the input drift x_t = x_{t-1} + sigma_t N(0,1)
    (sigma 0.3 -> 0.01) are drawn on the device from a seeded torch
    generator; (alpha, beta) ~ U(0.5,1.5) x U(0,0.01) per layer; tau is
    calibrated for ~60% NVFP4 from an all-INT8 run; TDC threshold 0.05,
    max_skip 1.  Also the PDR variant "pdr": max_skip 2 with a forced
    computed step every 4th step, and "measured_lines": (alpha, beta) refitted
    from E_rel measured on the first calib_steps steps (DMPQ calibration side)
    with tau set from them, "dmpq_tdc_fused_quant": DMPQ+TDC with the
    quantizing producers (LayerNorms and the up-projection's epilogue emit
    the next layer's NVFP4 / INT8 input; delayed NVFP4 scaling), and the
    "_mxcache" modes: the update cache stored as E4M3 codes with a
    power-of-two scale per 32 elements.  Timed: every step's graph replay
    plus its input copy.  modes: the subset of modes to run (None = all).
    Each mode also reports `roofline_frac`: the sum of its kernels' roofline
    times (stack_ideal_seconds, from the formats and skips it actually ran)
    over the measured time."""
    import torch
    from nvfp4_int8_mixed_gb300 import lib as _lib
    from nvfp4_int8_mixed_gb300.calibration import calibrate_lines, calibrate_tau
    from nvfp4_int8_mixed_gb300.stack import DiTStack
    sb_mx_bytes = lambda n: _lib().sixbit_mxcache_bytes(n)
    peaks, _ = load_peaks()
    fp4_peak = float(peaks["bf16_tflops"]) * FP4_OVER_BF16
    hbm = float(peaks["hbm_gbs"])
    c = STACKS[name]
    nb, M, H, F, T = c["n_blocks"], c["M"], c["H"], c["F"], c["steps"]
    gen = torch.Generator(device=dev).manual_seed(c["seed"])
    weights = []
    for _ in range(nb):
        weights.append({k: (torch.randn(shape, generator=gen, device=dev) * 0.02)
                        for k, shape in (("qkv", (3 * H, H)), ("out", (H, H)), ("up", (F, H)), ("down", (H, F)))})
    rng = np.random.default_rng(c["seed"])
    alpha = rng.uniform(0.5, 1.5, 4 * nb).astype(np.float32)
    beta = rng.uniform(0.0, 0.01, 4 * nb).astype(np.float32)
    x = torch.randn((M, H), generator=gen, device=dev)
    xs = [x.to(torch.bfloat16)]
    for t in range(1, T):
        x = x + synthetic.drift_sigma(t, T) * torch.randn((M, H), generator=gen, device=dev)
        xs.append(x.to(torch.bfloat16))
    del x
    stack = DiTStack(weights, alpha, beta, M, H, F, tau=0.0, tau_tdc=0.05, max_skip=1, device=dev, fused=True)
    stack.fused = False
    torch.cuda.synchronize()
    tau = calibrate_tau(stack, xs)
    res = {"config": f"{nb} blocks, M={M}, H={H}, F={F}, {T} steps", "tau": tau}
    runs = [("dmpq_tdc", 1, 0, None), ("dmpq_only", 0, 0, None), ("pdr_skip2_refresh4", 2, 4, None),
            ("dmpq_tdc_fused_quant", 1, 0, None), ("dmpq_tdc_mxcache", 1, 0, None),
            ("dmpq_tdc_fused_quant_mxcache", 1, 0, None)]
    if modes is not None:
        runs = [r for r in runs if r[0] in modes]
    if c.get("calib_steps") and (modes is None or "measured_lines" in modes):
        cal = calibrate_lines(stack, xs, weights, steps=c["calib_steps"])
        lines = (cal["alpha"].astype(np.float32), cal["beta"].astype(np.float32))
        fin = lambda a: float(np.nanmean(a))
        res["calibration"] = {"steps": c["calib_steps"], "e_rel_nvfp4_mean": fin(cal["e_rel_nvfp4"]),
                              "e_rel_int8_mean": fin(cal["e_rel_int8"]), "fit_r2_mean": fin(cal["r2"]),
                              "alpha_mean": fin(cal["alpha"]), "beta_mean": fin(cal["beta"]),
                              "delta_cos_mean": fin(cal["delta_cos"]), "delta_rel_mean": fin(cal["delta_rel"])}
        runs.append(("measured_lines", 1, 0, lines))
    res["bf16_torch_context"] = bf16_stack_context(weights, xs, H)
    if cpu_oracle:
        xb = xs[0].view(torch.int16).cpu().numpy().view(np.uint16)
        res["cpu_oracle"] = time_oracle_block({k: v.cpu().numpy() for k, v in weights[0].items()}, xb, M)
    del weights
    for mode, max_skip, refresh, lines in runs:
        stack.fused = "fused_quant" in mode
        stack.set_tdc_cache("mx" if mode.endswith("mxcache") else "bf16")
        if lines is not None:
            stack.alpha.copy_(torch.from_numpy(lines[0]))
            stack.beta.copy_(torch.from_numpy(lines[1]))
            tau = calibrate_tau(stack, xs)
            res["calibration"]["tau"] = tau
        stack.tau, stack.max_skip, stack.refresh_every = tau, max_skip, refresh
        stack.graph = None
        stack.reset()
        stack.capture()
        stack.reset()
        comp = torch.zeros(nb, dtype=torch.int32, device=dev)
        nv = torch.zeros(4 * nb, dtype=torch.int32, device=dev)      # NVFP4 flags of computed blocks
        nv_all = torch.zeros(4 * nb, dtype=torch.int32, device=dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for t in range(T):
            stack.x_in.copy_(xs[t])
            stack.step_dev.fill_(t)
            stack.graph.replay()
            cf = stack.cflag.int()
            comp += cf
            nv += stack.use_nvfp4.int() * cf.repeat_interleave(4)
            nv_all += stack.use_nvfp4.int()
        e1.record()
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) / 1e3
        comp_h = comp.cpu().numpy()
        nv_k = nv.view(nb, 4).sum(0).cpu().numpy()
        comp_total = int(comp_h.sum())
        kinds = ("qkv", "out", "up", "down")
        ideal = stack_ideal_seconds(M, H, F, {k: int(nv_k[i]) for i, k in enumerate(kinds)},
                                    {k: comp_total - int(nv_k[i]) for i, k in enumerate(kinds)},
                                    comp_total, nb * T - comp_total, fp4_peak, hbm)
        res[mode] = {"blocks_per_s": nb * T / sec, "ms_per_step": sec / T * 1e3,
                     "skipped_fraction": 1.0 - comp_total / (nb * T),
                     "nvfp4_fraction_after_step0": float(nv_all.sum()) / (4 * nb * (T - 1)),
                     "roofline_frac": ideal / sec, "roofline_ideal_ms_per_step": ideal / T * 1e3}
    # HBM footprint of the quantized stack vs a bf16 one (weights, TDC cache, block activations)
    w_params = nb * (3 * H * H + H * H + 2 * F * H)
    w_nvfp4 = sum(int(t.numel() * t.element_size()) for b in stack.wq for wl in b.values() for t in wl)
    act = sum(int(t.numel() * t.element_size()) for t in (stack.x_in, *stack.buf, stack.h1, stack.qkv, stack.x1,
                                                         stack.h2, stack.u, stack.codes, stack.sf, stack.planes))
    cache = nb * M * H * 2
    res["footprint_bytes"] = {"weights_nvfp4": w_nvfp4, "weights_bf16": 2 * w_params, "activations": act,
                              "tdc_cache": cache, "tdc_cache_mx": nb * int(sb_mx_bytes(M * H)),
                              "weights_ratio_bf16_over_nvfp4": 2 * w_params / w_nvfp4}
    del stack, xs
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------- our arm
def setup_gemm_set(sb, workload: str, dev):
    """Device inputs of one GEMM-set step (untimed): per layer the bf16
    activations (and residual), the weights quantized once, and the
    quantizer / GEMM outputs; plus a block input/output pair for the
    Gamma / DMPQ / TDC tail.  Seeds: 1 for the 2B set, 2 for the 5B set."""
    import torch
    layers = workload_layers(workload)
    M = synthetic.M_2B
    H = layers[0][1]
    seed = 1 if workload == "2b" else 2
    to_dev = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
    L, host_inputs = [], []
    for name, K, N, gelu, res in layers:
        lay = synthetic.gemm_layer(seed, M, K, N, res)
        x = to_dev(lay["a"])
        r = to_dev(lay["residual"]) if res else None
        wc, wsf, gw = sb.quantize_weight_nvfp4(torch.from_numpy(lay["w"]).to(dev))
        L.append(dict(name=name, K=K, N=N, gelu=gelu, x=x, r=r, wc=wc, wsf=wsf, gw=gw,
                      codes=torch.empty((M, K // 2), dtype=torch.uint8, device=dev),
                      sf=torch.empty(sb.sf_bytes(M, K), dtype=torch.uint8, device=dev),
                      ga=torch.empty(1, dtype=torch.float32, device=dev),
                      planes=torch.empty((3, M, K // 2), dtype=torch.uint8, device=dev),
                      s=torch.empty(M, dtype=torch.float32, device=dev),
                      y4=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                      y8=torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
        host_inputs.append((lay["a"], lay["residual"]))
    gp = synthetic.gamma_pair(7, M, H)
    tail = dict(bin=to_dev(gp["xin"]), bout=to_dev(gp["xout"]), delta=to_dev(gp["delta_prev"]),
                gamma=torch.zeros(4, dtype=torch.float32, device=dev),
                state=torch.tensor([1, 0], dtype=torch.int32, device=dev),
                step=torch.ones(1, dtype=torch.int32, device=dev),
                alpha=torch.linspace(0.5, 1.5, 4, device=dev), beta=torch.full((4,), 0.005, device=dev),
                lb=torch.zeros(4, dtype=torch.int32, device=dev), flags=torch.empty(4, dtype=torch.uint8, device=dev),
                gates=torch.empty((4, 2), dtype=torch.uint8, device=dev),
                cflag=torch.empty(1, dtype=torch.uint8, device=dev))
    tail["tdc_out"] = torch.empty_like(tail["bin"])
    sb.workspace(int(sb.lib().sixbit_workspace_size(M * H, 1)))
    return dict(L=L, M=M, H=H, layers=layers, tail=tail, gp=gp, host_inputs=host_inputs)


def gemm_set_step(sb, G):
    """step(evs=None, inp=None): one pass of the path over the set -- per layer
    tensor amax + NVFP4 quantize -> W4A4 GEMM, INT8 quantize -> W4A8 GEMM --
    then the Gamma/Delta pass, DMPQ and TDC.  evs: [launch][start, end]
    events recorded around every call; inp: device inputs to use instead of
    the defaults ({x, r: per layer, bin, bout})."""
    import torch
    L, T = G["L"], G["tail"]

    def step(evs=None, inp=None):
        cur = torch.cuda.current_stream()        # the capture stream while a graph is being captured
        k = 0
        ops = []
        for li, l in enumerate(L):
            x = inp["x"][li] if inp else l["x"]
            r = inp["r"][li] if inp else l["r"]
            ops += [
                lambda l=l, x=x: sb.quantize_act_nvfp4(x, out=(l["codes"], l["sf"], l["ga"])),
                lambda l=l, r=r: sb.qlinear_w4a4(l["codes"], l["sf"], l["ga"], l["wc"], l["wsf"], l["gw"], residual=r,
                                                 gelu=l["gelu"], out=l["y4"]),
                lambda l=l, x=x: sb.quantize_act_int8(x, out=(None, l["planes"], l["s"])),
                lambda l=l, r=r: sb.qlinear_w4a8(l["planes"], l["s"], l["wc"], l["wsf"], l["gw"], residual=r,
                                                 gelu=l["gelu"], out=l["y8"]),
            ]
        b_in, b_out = (inp["bin"], inp["bout"]) if inp else (T["bin"], T["bout"])
        g = T["gamma"]
        ops += [
            lambda: sb.block_gamma(b_in, b_out, delta=T["delta"], gamma_out=g[0:1], r2_out=g[1:2],
                                   tdc_state=T["state"]),
            lambda: sb.dmpq_assign(g[0:1], T["alpha"], T["beta"], T["lb"], 0.1, T["step"], use_nvfp4=T["flags"],
                                   gates=T["gates"]),
            lambda: sb.tdc_decide_and_apply(b_in, T["delta"], g[1:2], 0.05, 1, T["state"], T["cflag"], T["tdc_out"],
                                            gates=T["gates"]),
        ]
        for op in ops:
            if evs is not None:
                evs[k][0].record(cur)
            op()
            if evs is not None:
                evs[k][1].record(cur)
            k += 1

    names = []
    for l in L:
        names += [f"quant_nvfp4[{l['name']}]", f"w4a4[{l['name']}]", f"quant_int8[{l['name']}]", f"w4a8[{l['name']}]"]
    names += ["gamma_delta", "dmpq", "tdc"]
    return step, names


def time_gemm_set(sb, G, steps: int, warmup: int, ws: int, dev, clocks=False):
    """Time `steps` steps of the GEMM set: captured as one CUDA graph of the
    kernels alone, replayed once between CUDA events on the launching stream
    (barrier + synchronize on both sides, max over ranks).  Per-launch
    durations come from a second graph of the same steps with timing events
    around every launch, replayed after the timed region (median over the
    steps)."""
    import torch
    import torch.distributed as dist
    step, names = gemm_set_step(sb, G)
    for _ in range(max(warmup, 3)):
        step()
    sb.get_error()

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    try:
        torch.cuda.Event(enable_timing=True, external=True)
        mk_ev = lambda: torch.cuda.Event(enable_timing=True, external=True)
        in_graph_events = True
    except TypeError:
        in_graph_events = False
    evs = [[[mk_ev(), mk_ev()] for _ in names] for _ in range(steps)] if in_graph_events else None
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            step()
    graph_ev = None
    if in_graph_events:
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev):
            for i in range(steps):
                step(evs[i])
    sampler = None
    if clocks:
        props = torch.cuda.get_device_properties(dev)
        uuid = str(getattr(props, "uuid", ""))
        sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(dev.index)))
        time.sleep(0.3)
    stream = torch.cuda.current_stream()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    graph.replay()
    t1.record(stream)
    barrier()
    clk = sampler.stop() if sampler is not None else None
    sb.get_error()
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, ws, dev)
    n_ev = steps
    if graph_ev is not None:
        graph_ev.replay()
        torch.cuda.synchronize()
    else:
        n_ev = min(steps, 20)
        evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in names]
               for _ in range(n_ev)]
        for i in range(n_ev):
            step(evs[i])
        torch.cuda.synchronize()
    per = {n: [evs[i][k][0].elapsed_time(evs[i][k][1]) / 1e3 for i in range(n_ev)] for k, n in enumerate(names)}
    mean_t = {n: float(np.median(v)) for n, v in per.items()}
    del graph, graph_ev
    return dict(step=step, names=names, elapsed=elapsed, mean_t=mean_t, clocks=clk, in_graph_events=in_graph_events,
                launches_per_step=len(names) + len(G["L"]))   # + one tensor-amax pass per NVFP4 quantization


def gemm_set_report(G, T, fp4_peak: float, hbm: float, workload: str):
    """Per-kernel roofline figures of one timed GEMM set."""
    L, M, mean_t = G["L"], G["M"], T["mean_t"]
    gemm = {}
    for n in mean_t:
        if n.startswith("w4a"):
            l = L[[x["name"] for x in L].index(n.split("[")[1][:-1])]
            gemm[n] = gemm_roofline(n.split("[")[0], M, l["N"], l["K"], l["r"] is not None, mean_t[n], fp4_peak, hbm)
    bw = {}
    for l in L:
        for kind in ("nvfp4", "int8"):
            n = f"quant_{kind}[{l['name']}]"
            nb = quant_bytes(kind, M, l["K"])
            moved = nb if kind == "nvfp4" else (2 + 1.5) * M * l["K"] + 4 * M
            bw[n] = {"ms": mean_t[n] * 1e3, "bytes": nb, "GB/s": nb / mean_t[n] / 1e9,
                     "frac_hbm": nb / mean_t[n] / 1e9 / hbm,
                     "note": ("tensor amax pass + encode (two launches, no producer amax)" if kind == "nvfp4" else
                              f"writes the 3 E2M1 digit planes the W4A8 GEMM reads: {moved / nb:.3f}x the bytes")}
    nb = 8.0 * M * G["H"]
    bw["gamma_delta"] = {"ms": mean_t["gamma_delta"] * 1e3, "bytes": nb, "GB/s": nb / mean_t["gamma_delta"] / 1e9,
                         "frac_hbm": nb / mean_t["gamma_delta"] / 1e9 / hbm}
    pairs = {}
    for l in L:                                   # quantizer + GEMM back to back on one stream
        for kind, mode in (("nvfp4", "w4a4"), ("int8", "w4a8")):
            t = mean_t[f"quant_{kind}[{l['name']}]"] + mean_t[f"{mode}[{l['name']}]"]
            pairs[f"{mode}[{l['name']}]"] = {"ms": t * 1e3, "TFLOP/s": 2.0 * M * l["N"] * l["K"] / t / 1e12}
    return {"gemm": gemm, "bandwidth": bw, "quantizer_plus_gemm": pairs, "dmpq_ms": mean_t["dmpq"] * 1e3,
            "tdc_ms": mean_t["tdc"] * 1e3}


def _graph_launch_mean(fn, reps):
    """Mean duration of one launch: `reps` calls fn(0..reps-1) captured as one
    CUDA graph, the replay timed with CUDA events on the launching stream and
    divided by `reps` (median of 5 replays), so no host launch gap is inside."""
    import torch
    for i in range(3):
        fn(i)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(reps):
            fn(i)
    graph.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3 / reps)
    del graph
    return float(np.median(ts))


def time_quantizers_graph(sb, G, dev, reps=24):
    """Each activation quantizer alone, on each distinct K of the set: the
    NVFP4 encode pass with the tensor amax supplied (as a producer supplies
    it), and the INT8 quantizer writing the digit planes and row scales the
    W4A8 GEMM reads.  The launches rotate over copies of the activation whose
    total exceeds 300 MB, so each launch reads its input from HBM and no
    flush leaves dirty lines to be written back during a timed launch.  The
    per-launch figures of the step graph include its timing-event nodes;
    these do not."""
    peak = float(load_peaks()[0]["hbm_gbs"])
    nv, i8, seen = {}, {}, set()
    for l in G["L"]:
        if l["K"] in seen:
            continue
        seen.add(l["K"])
        nbuf = max(2, -(-(300 << 20) // (l["x"].numel() * 2)))
        xs = [l["x"]] + [l["x"].clone() for _ in range(nbuf - 1)]
        note = {"inputs": f"{nbuf} copies rotated ({nbuf * l['x'].numel() * 2 / 1e6:.0f} MB > L2)",
                "timing": f"graph of {reps} launches, per-launch mean"}
        amax, _ = sb.amax(l["x"])
        t = _graph_launch_mean(lambda i: sb.quantize_act_nvfp4(xs[i % nbuf], amax_in=amax,
                                                                out=(l["codes"], l["sf"], l["ga"])), reps)
        nb = quant_bytes("nvfp4", G["M"], l["K"])
        nv[f"K={l['K']}"] = {"us": t * 1e6, "GB/s": nb / t / 1e9, "frac_hbm": nb / t / 1e9 / peak, **note}
        t = _graph_launch_mean(lambda i: sb.quantize_act_int8(xs[i % nbuf], out=(None, l["planes"], l["s"])), reps)
        nb = quant_bytes("int8", G["M"], l["K"])
        i8[f"K={l['K']}"] = {"us": t * 1e6, "GB/s": nb / t / 1e9, "frac_hbm": nb / t / 1e9 / peak,
                             "bytes_note": "method's 3 B/element; the kernel writes 1.5 B of digit planes in place "
                                           "of the 1 B code", **note}
        sb.get_error()
        del xs
    return nv, i8


def time_gemms_graph(sb, G, fp4_peak, hbm, reps=10):
    """Each GEMM of the set alone: `reps` launches over rotated copies of its
    activation operand (more than 300 MB in all, so every launch reads it
    from HBM), captured as one CUDA graph; the per-launch mean, with the same
    roofline fields as the step's figures.  The step's per-launch figures
    include its timing-event nodes; these do not."""
    out = {}
    M = G["M"]
    for l in G["L"]:
        sb.quantize_act_nvfp4(l["x"], out=(l["codes"], l["sf"], l["ga"]))
        sb.quantize_act_int8(l["x"], out=(None, l["planes"], l["s"]))
        ops = {"w4a4": ((l["codes"], l["sf"]),
                        lambda a, l=l: sb.qlinear_w4a4(a[0], a[1], l["ga"], l["wc"], l["wsf"], l["gw"], residual=l["r"],
                                                       gelu=l["gelu"], out=l["y4"])),
               "w4a8": ((l["planes"], l["s"]),
                        lambda a, l=l: sb.qlinear_w4a8(a[0], a[1], l["wc"], l["wsf"], l["gw"], residual=l["r"],
                                                       gelu=l["gelu"], out=l["y8"]))}
        for mode, (a0, call) in ops.items():
            nb = sum(t.numel() * t.element_size() for t in a0)
            nbuf = max(2, -(-(300 << 20) // nb))
            bufs = [a0] + [tuple(t.clone() for t in a0) for _ in range(nbuf - 1)]
            t = _graph_launch_mean(lambda i: call(bufs[i % nbuf]), reps)
            r = gemm_roofline(mode, M, l["N"], l["K"], l["r"] is not None, t, fp4_peak, hbm)
            r["inputs"] = f"{nbuf} copies of the activation operand rotated ({nbuf * nb / 1e6:.0f} MB > L2)"
            out[f"{mode}[{l['name']}]"] = r
            del bufs
        sb.get_error()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import nvfp4_int8_mixed_gb300 as sb
    if not os.path.exists(sb.LIB_PATH):
        from nvfp4_int8_mixed_gb300 import build as _b
        _b.build()
    sb.lib()
    peaks, peak_kind = load_peaks()
    fp4_peak = float(peaks["bf16_tflops"]) * FP4_OVER_BF16
    hbm = float(peaks["hbm_gbs"])

    # ---- headline workload: setup (untimed), then the K timed steps
    G = setup_gemm_set(sb, args.workload, dev)
    L, M, layers = G["L"], G["M"], G["layers"]
    flops_layer = [2 * M * l["N"] * l["K"] for l in L]
    flops_step = 2 * sum(flops_layer)
    T = time_gemm_set(sb, G, args.steps, args.warmup, ws, dev, clocks=True)
    elapsed, mean_t, step = T["elapsed"], T["mean_t"], T["step"]
    in_graph, launches_step, clocks = T["in_graph_events"], T["launches_per_step"], T["clocks"]
    value = job_throughput(flops_step * args.steps, ws, elapsed) / 1e12
    stream = torch.cuda.current_stream()

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- end to end through the public API: pinned host inputs copied in every step
    tl = G["tail"]
    pinned = []
    h2d = 0
    for (a, r), l in zip(G["host_inputs"], L):
        ha = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
        hr = torch.from_numpy(r.view(np.int16)).view(torch.bfloat16).pin_memory() if r is not None else None
        pinned.append((ha, hr))
        h2d += ha.numel() * 2 + (hr.numel() * 2 if hr is not None else 0)
    hb = [torch.from_numpy(G["gp"][k].view(np.int16)).view(torch.bfloat16).pin_memory() for k in ("xin", "xout")]
    h2d += sum(t.numel() * 2 for t in hb)
    res_host = torch.empty(4 + 4 + 1, dtype=torch.uint8).pin_memory()
    out_host = torch.empty(2, dtype=torch.float32).pin_memory()
    d2h = res_host.numel() + out_host.numel() * 4

    # Inputs are double-buffered on the device: while the compute stream runs
    # step s on one set, two copy streams bring step s+1's inputs into the
    # other.  Every step copies all of its inputs from pinned host memory and
    # reads its decisions back inside the timed region; events order a set's
    # copies after the step that last read it.
    sets = [dict(x=[l["x"] for l in L], r=[l["r"] for l in L], bin=tl["bin"], bout=tl["bout"]),
            dict(x=[torch.empty_like(l["x"]) for l in L],
                 r=[torch.empty_like(l["r"]) if l["r"] is not None else None for l in L],
                 bin=torch.empty_like(tl["bin"]), bout=torch.empty_like(tl["bout"]))]
    copy_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    ready = [[torch.cuda.Event() for _ in copy_streams] for _ in sets]
    free = [torch.cuda.Event() for _ in sets]

    def load(si, after=None):
        d = sets[si]
        jobs = []
        for li, (ha, hr) in enumerate(pinned):
            jobs.append((d["x"][li], ha))
            if hr is not None:
                jobs.append((d["r"][li], hr))
        jobs += [(d["bin"], hb[0]), (d["bout"], hb[1])]
        load_bytes = [0] * len(copy_streams)
        for cs in copy_streams:
            cs.wait_event(free[si])                # the step that last read this set is done
            if after is not None:
                cs.wait_event(after)
        for dst, src in sorted(jobs, key=lambda j: -j[1].numel()):
            c = load_bytes.index(min(load_bytes))  # balance bytes over the copy streams
            with torch.cuda.stream(copy_streams[c]):
                dst.copy_(src, non_blocking=True)
            load_bytes[c] += src.numel() * src.element_size()
        for c, cs in enumerate(copy_streams):
            ready[si][c].record(cs)

    def e2e_step(s, last):
        si = s % 2
        for ev in ready[si]:
            stream.wait_event(ev)
        step(inp=sets[si])
        free[si].record(stream)
        out_host.copy_(tl["gamma"][0:2], non_blocking=True)
        res_host[0:4].copy_(tl["flags"], non_blocking=True)
        res_host[4:8].copy_(tl["gates"].view(-1)[0:4], non_blocking=True)
        res_host[8:9].copy_(tl["cflag"], non_blocking=True)
        if not last:
            load((s + 1) % 2)

    e2e_steps = max(3, args.steps // 4)
    load(0)                                        # untimed warm-up of the pipeline
    for s in range(2):
        e2e_step(s, last=(s == 1))
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    load(0, after=e0)                              # the first step's copies are inside the timed region
    for s in range(e2e_steps):
        e2e_step(s, last=(s == e2e_steps - 1))
    e1.record(stream)
    barrier()
    e2e_elapsed = max_over_ranks(e0.elapsed_time(e1) / 1e3, ws, dev)
    e2e_value = job_throughput(flops_step * e2e_steps, ws, e2e_elapsed) / 1e12
    del sets, pinned

    # ---- roofline of the dominant kernel: the longest launch of the step,
    # its method FLOPs (2MNK) against the dense FP4 tensor peak
    report = gemm_set_report(G, T, fp4_peak, hbm, args.workload)
    gemm_names = [n for n in T["names"] if n.startswith("w4a")]
    dom = max(gemm_names, key=lambda n: mean_t[n])
    dr = report["gemm"][dom]
    traffic = dram_traffic(dom) if args.workload == "2b" else None
    roofline = {"bound": "tensor", "kernel": dom, "achieved": dr["TFLOP/s"], "peak": fp4_peak, "unit": "TFLOP/s",
                "frac": dr["TFLOP/s"] / fp4_peak, "traffic": traffic,
                "peak_note": f"dense FP4 tensor peak: {peak_kind} bf16 burst {peaks['bf16_tflops']} TFLOP/s x the "
                             f"nominal FP4/BF16 ratio 6; achieved = the method's 2MNK / the launch's median time"}
    if dom.startswith("w4a8"):
        roofline["fp4_pipe_frac"] = dr["fp4_pipe_frac"]
        roofline["fp4_pipe_note"] = ("W4A8 issues three exact E2M1 digit-plane MMAs per product on the FP4 pipe: "
                                     "3 x achieved / peak is that pipe's busy fraction; its design ceiling is peak/3")
    w4a4 = {n: v["frac_fp4_peak"] for n, v in report["gemm"].items() if n.startswith("w4a4")}

    extra = {}
    if rank == 0 and args.workload == "2b":
        extra["quantizing_producers"] = time_producers(sb, L, dev, (tl["bin"], tl["bout"]))
        extra["quant_nvfp4_amax_given"], extra["quant_int8_graph"] = time_quantizers_graph(sb, G, dev)
        extra["gemm_graph"] = time_gemms_graph(sb, G, fp4_peak, hbm)
    del G, T
    torch.cuda.empty_cache()

    # ---- the 5B-class GEMM set (quantizer and GEMM timed separately and back to back)
    set5 = None
    if rank == 0 and args.workload == "2b" and not args.no_5b:
        G5 = setup_gemm_set(sb, "5b", dev)
        T5 = time_gemm_set(sb, G5, args.steps, args.warmup, 1, dev)
        f5 = 2 * sum(2 * G5["M"] * l["N"] * l["K"] for l in G5["L"])
        rep5 = gemm_set_report(G5, T5, fp4_peak, hbm, "5b")
        set5 = {"config": workload_config("5b", G5["M"], G5["layers"], 1)["workload"],
                "value": f5 * args.steps / T5["elapsed"] / 1e12, "unit": "TFLOP/s",
                "ms_per_step": T5["elapsed"] / args.steps * 1e3, "per_kernel": rep5}
        del G5, T5
        torch.cuda.empty_cache()

    stacks = {}
    if rank == 0 and args.stack != "none":
        stacks["2b"] = run_stack_bench(args.stack, dev, cpu_oracle=not args.no_cpu_baseline)
        if args.stack == "2b" and not args.no_5b:
            stacks["5b_cfg"] = run_stack_bench("5b", dev, cpu_oracle=False, modes=("dmpq_tdc", "dmpq_only"))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rows, cols = 64, 512
        v_cpu, dt_cpu, fl = time_oracle(layers, M, rows, cols, steps=1, warmup=0, seed=1)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{rows} random rows x {cols} random output columns of each of the 4 layers, NVFP4+W4A4 and "
                         f"INT8+W4A8 ({fl / 1e9:.1f} GFLOP, {dt_cpu:.1f} s), plus Gamma/DMPQ/TDC on a 64x1920 pair"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
                "warmup": max(args.warmup, 3), "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "fp4 (e2m1 x e2m1, fp32 accumulate)",
                "data": "synthetic",
                "config": dict(workload_config(args.workload, M, layers, ws),
                               timing="the K steps captured as one CUDA graph, replayed once between CUDA events; "
                                      + ("per-launch durations from a second, instrumented graph of the same steps"
                                         if in_graph else "per-launch events from eager steps")),
                "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                        "d2h_bytes_per_step": int(d2h),
                        "d2h_note": "the step's decisions (Gamma, r2, DMPQ flags and gates, TDC compute bit) are read "
                                    "back; the eight GEMM outputs stay in device memory, where the next layer of the "
                                    "network would read them"},
                "gpu_launches": launches_step * args.steps,
                "clocks": clocks, "roofline": roofline, "w4a4_frac_fp4_peak": w4a4,
                "cpu_baseline": cpu,
                "gemm_set_5b": set5,
                "dit_stack": stacks.get("2b"), "dit_stack_5b_cfg": stacks.get("5b_cfg"),
                "per_kernel": dict(report, **extra)}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["2b", "5b"], default="2b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stack", choices=["2b", "5b", "none"], default="2b",
                    help="DiT block stack measured after the GEMM-set step (blocks/s with DMPQ+TDC)")
    ap.add_argument("--no-5b", action="store_true",
                    help="skip the 5B-class GEMM set and the 5B CFG stack that the default run also measures")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
