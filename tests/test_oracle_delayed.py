"""Pins of delayed NVFP4 scaling (quantization inside the producing kernel)
and of the fused-producer stack rule: the zero history, the power-of-two
headroom identity, the saturation bound, and convergence to the dynamic
result at a fixed input."""
import numpy as np

import synthetic
from oracle import block, codecs, nvfp4


def _x(seed=0, R=64, K=256, scale=1.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((R, K)) * scale).astype(np.float32)
    return codecs.bf16_to_f32(codecs.f32_to_bf16(x))


def test_zero_history_gives_zero_codes():
    x = _x()
    codes, sf, g, used, new = nvfp4.quantize_delayed(x, 0.0)
    assert used == 0 and g == 1.0 and not codes.any() and not sf.any()
    assert new == np.max(np.abs(x))


def test_power_of_two_headroom_keeps_the_dequantized_tensor():
    # amax unchanged: S_b halves and g doubles exactly, so S_b * g and the codes are those of the dynamic path
    x = _x(1)
    ref_c, ref_sf, ref_g, amax = nvfp4.quantize(x)
    for h in (2.0, 4.0):
        c, sf, g, used, _ = nvfp4.quantize_delayed(x, amax, h)
        assert used == h * amax and g == h * ref_g
        assert np.array_equal(c, ref_c)
        S, S_ref = codecs.e4m3_decode(sf), codecs.e4m3_decode(ref_sf)
        assert np.array_equal(S * h, S_ref)
        assert np.array_equal(nvfp4.dequantize(c, sf, g), nvfp4.dequantize(ref_c, ref_sf, ref_g))


def test_grown_amax_saturates_at_the_used_amax():
    x0 = _x(2)
    a0 = np.max(np.abs(x0))
    x1 = codecs.bf16_to_f32(codecs.f32_to_bf16(3.0 * x0))      # amax grew 3x, past headroom 2
    c, sf, g, used, new = nvfp4.quantize_delayed(x1, a0, 2.0)
    d = nvfp4.dequantize(c, sf, g)
    assert used == 2 * a0 and new == np.max(np.abs(x1))
    assert np.max(np.abs(d)) == 2688.0 * float(g)              # saturated blocks: 6 * 448 * g
    assert abs(2688.0 * float(g) - used) <= used * 2.0 ** -23  # = amax_used up to g's rounding
    small = np.max(np.abs(x1.reshape(64, -1, 16)), axis=2) < used / 2
    # blocks well inside the range keep the dynamic path's precision: error below half an E2M1 step
    err = np.abs(d - x1).reshape(64, -1, 16)[small]
    S = codecs.e4m3_decode(sf).astype(np.float64)[small][:, None] * float(g)
    assert np.all(err <= S * 1.0 + 1e-12)


def _setup(nb=1, M=48, H=64, F=128, steps=6, seed=5):
    st = synthetic.stack_setup(seed, nb, H, F)
    wq = [{k: block.quantize_weights(v) for k, v in b.items()} for b in st["blocks"]]
    xs = synthetic.stack_inputs(st["noise_seed"], M, H, 2)
    return st, wq, xs


def test_block_converges_to_dynamic_at_fixed_input():
    # three fused producers in a chain (h1 -> h2 -> u): from the fourth call on
    # every history entry is the exact amax of the same input, and with the
    # power-of-two headroom the block equals the dynamic one bit for bit
    st, wq, xs = _setup()
    flags = np.ones(4, np.uint8)
    ref = block.block_forward(xs[0], wq[0], flags)
    hist = np.zeros(3, np.float32)
    outs = [block.block_forward(xs[0], wq[0], flags, hist) for _ in range(5)]
    assert not np.array_equal(outs[0], ref)                    # zero history: codes 0 in all three layers
    assert np.array_equal(outs[3], ref) and np.array_equal(outs[4], ref)
    h1 = block.layernorm(xs[0])
    assert hist[0] == np.max(np.abs(codecs.bf16_to_f32(h1)))


def test_int8_layers_are_unchanged_by_fusion():
    st, wq, xs = _setup()
    flags = np.zeros(4, np.uint8)
    hist = np.zeros(3, np.float32)
    assert np.array_equal(block.block_forward(xs[0], wq[0], flags, hist), block.block_forward(xs[0], wq[0], flags))
    assert (hist > 0).all()                                    # the history is recorded whatever the format


def test_stack_skipped_block_keeps_its_history():
    st, wq, xs = _setup()
    steps = 6
    x = [xs[0]] * steps
    flags = [np.ones(4, np.uint8)] * steps
    skips = [np.array([1 if t == 2 else 0], np.uint8) for t in range(steps)]
    r = block.run_stack(x, wq, st["alpha"], st["beta"], 0.0, 0.0, 1, forced_flags=flags, forced_skips=skips,
                        fused=True)
    ref = block.block_forward(xs[0], wq[0], np.ones(4, np.uint8))
    # computed calls at steps 0, 1, 3, 4, 5: the fourth computed call is step 4
    assert np.array_equal(r["outputs"][4], ref) and np.array_equal(r["outputs"][5], ref)
    assert np.array_equal(r["amax_hist"][2], r["amax_hist"][1])
    assert len(r["amax_hist"]) == steps


def test_fused_stack_matches_unfused_once_histories_settle():
    st, wq, xs = _setup(nb=2)
    steps = 8
    x = [xs[0]] * steps
    flags = [np.ones(8, np.uint8)] * steps
    a = block.run_stack(x, wq, st["alpha"], st["beta"], 0.0, 0.0, 1, use_tdc=False, forced_flags=flags, fused=True)
    b = block.run_stack(x, wq, st["alpha"], st["beta"], 0.0, 0.0, 1, use_tdc=False, forced_flags=flags)
    # block 0 settles after 3 calls, block 1 (whose input settles at step 3) after 3 more
    assert np.array_equal(a["outputs"][6], b["outputs"][6]) and np.array_equal(a["outputs"][7], b["outputs"][7])
