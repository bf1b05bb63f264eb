"""Pins of the synthetic block pieces (LayerNorm vs torch) and properties of
the small stack that follow from the method's rules."""
import numpy as np
import torch

import synthetic
from oracle import block, codecs


def test_layernorm_vs_torch():
    rng = np.random.default_rng(0)
    x = codecs.f32_to_bf16(rng.standard_normal((17, 96)).astype(np.float32) * 3 + 1)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(codecs.bf16_to_f32(x).astype(np.float64)), (96,), eps=1e-5)
    assert np.array_equal(block.layernorm(x), codecs.f64_to_bf16(ref.numpy()))


def _tiny_stack(steps=5, nb=3, M=40, H=64, F=128, seed=7):
    st = synthetic.stack_setup(seed, nb, H, F)
    wq = [{k: block.quantize_weights(v) for k, v in b.items()} for b in st["blocks"]]
    xs = synthetic.stack_inputs(st["noise_seed"], M, H, steps)
    return st, wq, xs


def test_stack_tdc_off_equals_zero_threshold():
    st, wq, xs = _tiny_stack()
    a = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.05, 0.0, 1, use_tdc=True)
    b = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.05, 0.05, 1, use_tdc=False)
    for x, y in zip(a["outputs"], b["outputs"]):
        assert np.array_equal(x, y)
    assert not np.any(a["skips"])


def test_stack_flags_follow_gamma_and_uniform_extremes():
    st, wq, xs = _tiny_stack(steps=3)
    r = block.run_stack(xs, wq, st["alpha"], st["beta"], np.inf, 0.0, 1)
    assert not r["flags"][0].any() and all(f.all() for f in r["flags"][1:])
    forced = [np.ones(12, np.uint8)] * 3
    forced[0] = np.zeros(12, np.uint8)
    r2 = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.0, 0.0, 1, forced_flags=forced)
    for x, y in zip(r["outputs"], r2["outputs"]):
        assert np.array_equal(x, y)


def test_stack_skip_reuses_delta():
    st, wq, xs = _tiny_stack(steps=6)
    r = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.05, 10.0, 1)   # huge tau_tdc: skip when allowed
    skips = np.array(r["skips"])
    assert not skips[:2].any()                     # need two fresh updates first
    assert skips[2].all() and not skips[3].any() and skips[4].all()   # max_skip = 1 alternates


def test_stack_periodic_refresh_computes_every_kth_step():
    st, wq, xs = _tiny_stack(steps=8)
    r = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.05, 10.0, 3, refresh_every=3)
    skips = np.array(r["skips"])
    assert not skips[[0, 3, 6]].any()              # refresh steps are computed
    assert skips[2].all() and skips[4].all() and skips[5].all() and skips[7].all()


def test_block_residual_wiring_with_zero_weights():
    # all weights zero: every linear outputs 0 (+ residual), GELU(0) = 0, so out == in exactly
    rng = np.random.default_rng(3)
    H, F, M = 64, 128, 24
    x = codecs.f32_to_bf16(rng.standard_normal((M, H)).astype(np.float32))
    zero = lambda n, k: block.quantize_weights(np.zeros((n, k), np.float32))
    wq = dict(qkv=zero(3 * H, H), out=zero(H, H), up=zero(F, H), down=zero(H, F))
    for flags in ([0, 0, 0, 0], [1, 1, 1, 1], [1, 0, 1, 0]):
        assert np.array_equal(block.block_forward(x, wq, flags), x)


def test_block_out_proj_reads_the_v_slice():
    # weights only in the Q and K rows of W_qkv: the V slice is zero, so x1 = x and
    # with W_up = 0 the block is the identity; weights in the V rows change the output
    rng = np.random.default_rng(4)
    H, F, M = 64, 128, 24
    x = codecs.f32_to_bf16(rng.standard_normal((M, H)).astype(np.float32))
    w_qk = np.zeros((3 * H, H), np.float32)
    w_qk[:2 * H] = rng.standard_normal((2 * H, H)).astype(np.float32)
    w_v = np.zeros((3 * H, H), np.float32)
    w_v[2 * H:] = rng.standard_normal((H, H)).astype(np.float32)
    eye = block.quantize_weights(np.eye(H, dtype=np.float32))
    zero = lambda n, k: block.quantize_weights(np.zeros((n, k), np.float32))
    base = dict(out=eye, up=zero(F, H), down=zero(H, F))
    out_qk = block.block_forward(x, dict(base, qkv=block.quantize_weights(w_qk)), [1, 1, 1, 1])
    out_v = block.block_forward(x, dict(base, qkv=block.quantize_weights(w_v)), [1, 1, 1, 1])
    assert np.array_equal(out_qk, x)
    assert not np.array_equal(out_v, x)


def test_chunked_weight_quantization_and_dequantized_cache_change_nothing():
    rng = np.random.default_rng(3)
    w = (0.02 * rng.standard_normal((300, 128))).astype(np.float32)
    full = block.quantize_weights(w)
    chunked = block.quantize_weights(w, chunk_rows=128, keep_dequantized=True)
    assert np.array_equal(full["codes"], chunked["codes"]) and np.array_equal(full["sf"], chunked["sf"])
    assert full["g"] == chunked["g"]
    h = codecs.f32_to_bf16(rng.standard_normal((9, 128)).astype(np.float32))
    for nv in (True, False):
        assert np.array_equal(block.qlinear(h, full, nv, gelu=True), block.qlinear(h, chunked, nv, gelu=True))


def test_block_on_a_row_subset_with_the_full_tensor_amaxes():
    # Only the NVFP4 tensor amaxes couple the rows of a block: given the
    # whole tensors' amaxes, a row subset reproduces those rows exactly.
    from oracle import nvfp4
    st = synthetic.stack_setup(5, 1, 64, 128)
    wq = {k: block.quantize_weights(v) for k, v in st["blocks"][0].items()}
    x = synthetic.stack_inputs(st["noise_seed"], 96, 64, 1)[0]
    flags = np.array([1, 1, 1, 1], np.uint8)
    full = block.block_forward(x, wq, flags)
    # the full block's layer inputs, rebuilt step by step to take their amaxes
    h1 = block.layernorm(x)
    qkv = block.qlinear(h1, wq["qkv"], True)
    v = np.ascontiguousarray(qkv[:, 128:192])
    x1 = block.qlinear(v, wq["out"], True, residual=x)
    h2 = block.layernorm(x1)
    u = block.qlinear(h2, wq["up"], True, gelu=True)
    amax = [nvfp4.tensor_amax(codecs.bf16_to_f32(t)) for t in (h1, v, h2, u)]
    rows = np.array([0, 7, 50, 95])
    sub = block.block_forward(x[rows], wq, flags, layer_amax=amax)
    assert np.array_equal(sub, full[rows])
    # without them the subset takes its own (smaller) amaxes and differs
    assert not np.array_equal(block.block_forward(x[rows], wq, flags), full[rows])
