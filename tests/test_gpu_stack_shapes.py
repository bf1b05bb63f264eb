"""GPU parity of the DiT stack at the shapes of the two stack workloads:
the 2B-class block (M = 17776 tokens, hidden 1920, FFN 7680) and the
5B-class classifier-free-guidance block (M = 2 x 17776, hidden 3072, FFN
12288).

One block at each shape runs through the library with a forced mix of
NVFP4 and INT8 layers.  Each layer's device output is compared, on sampled
rows, with the oracle's layer applied to the device's own layer input; the
NVFP4 tensor amax the oracle quantizes with is its own maximum over the
whole device tensor.  The block output is compared with the oracle's block
run on the sampled rows (relative L2 <= 2e-3).

Then two steps of the 30-block 2B-class stack (DMPQ and TDC active; the 30
blocks share one set of weights so the oracle quantizes them once): every
block against the oracle's block on the device's own block input, and the
free-running chain against the oracle's chain on the sampled rows, under
the device's decisions."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import block as o_block, codecs, dmpq as o_dmpq, nvfp4 as o_nvfp4
from tests.helpers import assert_gemm_close, dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu

SHAPES = {"2b": (synthetic.M_2B, 1920, 7680), "5b_cfg": (2 * synthetic.M_2B, 3072, 12288)}
_cache = {}


def _weights(name):
    """Weights N(0, 0.02) of one block at the shape, and the oracle's NVFP4
    quantization of them (with the decoded matrices kept for many products)."""
    if name not in _cache:
        M, H, F = SHAPES[name]
        g = synthetic.rng(40 + len(name))
        w = dict(qkv=synthetic.weights(g, 3 * H, H), out=synthetic.weights(g, H, H),
                 up=synthetic.weights(g, F, H), down=synthetic.weights(g, H, F))
        wq = {k: o_block.quantize_weights(v, chunk_rows=1024, keep_dequantized=True) for k, v in w.items()}
        _cache[name] = (w, wq)
    return _cache[name]


def _amax(bits):
    return o_nvfp4.tensor_amax(codecs.bf16_to_f32(bits))


def _rows(M, n, seed):
    r = np.random.default_rng(seed).choice(M, n, replace=False)
    return np.unique(np.concatenate([r, [0, M - 1]]))          # includes the ragged last row tile


def _rel_l2(got_bits, ref_bits):
    g = codecs.bf16_to_f32(got_bits).astype(np.float64)
    r = codecs.bf16_to_f32(ref_bits).astype(np.float64)
    return float(np.linalg.norm(g - r) / np.linalg.norm(r))


@pytest.mark.parametrize("name,flags", [("2b", (1, 0, 1, 0)), ("2b", (0, 1, 0, 1)),
                                        ("5b_cfg", (1, 0, 1, 0)), ("5b_cfg", (0, 1, 0, 1))])
def test_one_block_at_full_shape_layer_by_layer(name, flags):
    from nvfp4_int8_mixed_gb300.stack import DiTStack
    M, H, F = SHAPES[name]
    w, wq = _weights(name)
    # DMPQ forced through its own rule: alpha = 0, beta 0 (NVFP4) or 1 (INT8), tau 0.5
    beta = np.array([0.0 if f else 1.0 for f in flags], np.float32)
    stack = DiTStack([w], np.zeros(4, np.float32), beta, M, H, F, tau=0.5, tau_tdc=0.0, max_skip=0)
    xs = synthetic.stack_inputs(50 + len(name), M, H, 2)
    cap = {}
    for t in range(2):                           # step 0 runs all-INT8; step 1 takes the forced mix
        stack.x_in.copy_(dev_bf16(xs[t]))
        stack.step_dev.fill_(t)
        stack.enqueue_step(hook=(lambda l, i, x: cap.__setitem__(i, x.clone())) if t == 1 else None)
    torch.cuda.synchronize()
    assert host(stack.use_nvfp4).tolist() == list(flags)
    x = xs[1]
    h1, v, h2, u = (host_bf16_bits(cap[i]) for i in range(4))
    qkv, x1, out = host_bf16_bits(stack.qkv), host_bf16_bits(stack.x1), host_bf16_bits(stack.out)
    del cap, stack
    torch.cuda.empty_cache()
    amax = [_amax(t) for t in (h1, v, h2, u)]
    R = _rows(M, 30, M + H)
    # LayerNorms: within one bf16 rounding of the oracle's
    for got, src in ((h1, x), (h2, x1)):
        ref = codecs.bf16_to_f32(o_block.layernorm(src[R])).astype(np.float64)
        assert np.all(np.abs(codecs.bf16_to_f32(got[R]) - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-6)
    # each linear layer on the device's own input, at the GEMM tolerance
    layers = ((h1, "qkv", 0, False, None, qkv), (v, "out", 1, False, x, x1), (h2, "up", 2, True, None, None),
              (u, "down", 3, False, x1, out))
    for inp, k, i, gelu, res, got in layers:
        ref = o_block.qlinear(inp[R], wq[k], bool(flags[i]), gelu=gelu, residual=None if res is None else res[R],
                              amax_t=amax[i])
        got_rows = (u if k == "up" else got)[R]
        assert_gemm_close(codecs.bf16_to_f32(got_rows), codecs.bf16_to_f32(ref), "bf16")
    # the block on the sampled rows: the oracle's own chain, the device's tensor amaxes only as scalars
    ref_out = o_block.block_forward(x[R], wq, np.array(flags, np.uint8), layer_amax=amax)
    assert _rel_l2(out[R], ref_out) <= 2e-3


def test_30_block_stack_two_free_running_steps_at_2b_shape():
    """Every block, given the device's own block input rows and layer amaxes,
    matches the oracle's block to 2e-3 (teacher forcing per block, both
    steps): the parity check.  Free running, the two sides' independent bf16
    roundings flip a few NVFP4 / INT8 codes in the next block, so their
    divergence grows with depth: it is held to 2e-3 over the first three
    blocks (the depth of the small stack test) and after that to at most
    linear growth, 2e-3 * depth / 3 (observed on GB300: 6.4e-3 after 29
    blocks of the mixed step)."""
    from nvfp4_int8_mixed_gb300.stack import DiTStack
    M, H, F = SHAPES["2b"]
    nb, steps = 30, 2
    w, wq = _weights("2b")
    g = synthetic.rng(61)
    alpha = g.uniform(0.5, 1.5, 4 * nb).astype(np.float32)
    beta = g.uniform(0.0, 0.01, 4 * nb).astype(np.float32)
    stack = DiTStack([w] * nb, alpha, beta, M, H, F, tau=0.0, tau_tdc=0.05, max_skip=1)
    xs = synthetic.stack_inputs(62, M, H, steps)
    R = _rows(M, 14, 63)
    amax, blk = {}, {}

    def hook(t):
        def f(l, i, x):
            amax[(t, l, i)] = _amax(host_bf16_bits(x))   # the oracle's max over the whole device tensor
        return f

    def block_hook(t):
        def f(l, h, out):
            blk[(t, l)] = (host_bf16_bits(h)[R], host_bf16_bits(out)[R])
        return f

    flags, skips = [], []
    lb = np.repeat(np.arange(nb), 4)
    for t in range(steps):
        if t == 1:                                       # tau: the median prediction from step 0's Gamma
            p = o_dmpq.predict(host(stack.gamma), alpha, beta, lb)
            stack.tau = float(np.median(p))
        stack.x_in.copy_(dev_bf16(xs[t]))
        stack.step_dev.fill_(t)
        stack.enqueue_step(hook=hook(t), block_hook=block_hook(t))
        torch.cuda.synchronize()
        flags.append(host(stack.use_nvfp4).copy())
        skips.append(1 - host(stack.cflag))
    assert not any(s.any() for s in skips)              # two steps: TDC has no two fresh updates yet
    assert 0 < flags[1].sum() < 4 * nb                   # a real NVFP4 / INT8 mix at step 1
    for t in range(steps):
        h = xs[t][R]
        for l in range(nb):
            f = flags[t][4 * l:4 * l + 4]
            la = [amax[(t, l, i)] for i in range(4)]
            h_in, out = blk[(t, l)]
            forced = o_block.block_forward(h_in, wq, f, layer_amax=la)
            assert _rel_l2(out, forced) <= 2e-3, ("teacher-forced", t, l, _rel_l2(out, forced))
            h = o_block.block_forward(h, wq, f, layer_amax=la)
            d = _rel_l2(out, h)
            assert d <= 2e-3 * max(1.0, (l + 1) / 3), ("free-running", t, l, d)
