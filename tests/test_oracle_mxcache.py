"""Pins of the compressed TDC cache (E4M3 codes, one power-of-two scale per
32 elements) and of the Gamma / TDC rules that use it."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import block, codecs, gamma, mxcache, tdc


def _bf16(x):
    return codecs.bf16_to_f32(codecs.f32_to_bf16(np.asarray(x, np.float32)))


def test_grid_values_round_trip():
    # every finite positive E4M3 magnitude times 2^k, in blocks whose maximum is 448 * 2^k
    mags = codecs.e4m3_decode(np.arange(0x7F)).astype(np.float64)           # codes 0x00 .. 0x7E
    vals = np.concatenate([mags, -mags[1:], np.zeros(256 - (2 * len(mags) - 1))])
    for k in (-20, -3, 0, 5, 30):
        v = (vals * 2.0 ** k).astype(np.float32)
        blocks = v.reshape(-1, 32)
        blocks[:, 0] = 448 * 2.0 ** k                                        # scale k in every block
        codes, sc = mxcache.encode(blocks.reshape(-1))
        assert (sc == k + 127).all()
        assert np.array_equal(mxcache.decode(codes, sc), blocks.reshape(-1))


def test_scale_boundary_and_powers_of_two():
    for k in (-8, 0, 3):
        at = np.float32(448 * 2.0 ** k)
        above = np.nextafter(at, np.float32(np.inf))                         # needs one more binade
        assert mxcache.scale_exponent([at])[0] == k
        assert mxcache.scale_exponent([above])[0] == k + 1
    for j in range(-30, 31, 7):                                              # A = 2^j: 2^j <= 1.75 * 2^(k+8) from k = j-8
        assert mxcache.scale_exponent([2.0 ** j])[0] == j - 8
    assert mxcache.scale_exponent([0.0])[0] == -127


def test_zero_block():
    codes, sc = mxcache.encode(np.zeros(64, np.float32))
    assert not codes.any() and (sc == 0).all() and not mxcache.decode(codes, sc).any()


def test_codes_match_torch_float8_and_error_bound():
    rng = np.random.default_rng(3)
    v = _bf16(rng.standard_normal(32 * 400) * np.repeat(np.exp2(rng.integers(-12, 12, 400)), 32))
    v[:64] = _bf16(rng.standard_normal(64) * 1e-3)                           # small blocks
    codes, sc = mxcache.encode(v)
    k = sc.astype(np.int64) - 127
    scaled = (v.reshape(-1, 32).astype(np.float64) * np.exp2(-k)[:, None]).astype(np.float32)
    ref = torch.from_numpy(scaled.reshape(-1)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)
    d = mxcache.decode(codes, sc).astype(np.float64)
    s = np.abs(scaled.reshape(-1).astype(np.float64))
    step = np.where(s >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(s, 2.0 ** -6))) - 3), 2.0 ** -9)
    bound = 0.5 * step * np.repeat(np.exp2(k), 32)
    assert np.all(np.abs(d - v) <= bound)                                    # half a step: no block is clipped
    assert np.all(np.abs(scaled) <= 448)


def test_layout_codes_then_scales():
    v = _bf16(np.arange(64, dtype=np.float32) - 20)
    codes, sc = mxcache.encode(v)
    b = mxcache.to_bytes(codes, sc)
    assert b.size == 66 and np.array_equal(b[:64], codes) and np.array_equal(b[64:], sc)


def test_gamma_pass_with_cached_update():
    rng = np.random.default_rng(5)
    n = 32 * 8
    xin = codecs.f32_to_bf16(np.zeros(n, np.float32))
    prev = mxcache.roundtrip_bf16(codecs.f32_to_bf16(rng.standard_normal(n).astype(np.float32)))
    out = codecs.f32_to_bf16(prev)                  # cached values are E4M3 * 2^k: exact in bf16
    g, dn, r2 = gamma.block_pass(xin, out, prev, computed=True, cache="mx")
    assert r2 == 0 and np.array_equal(dn, prev)      # Delta_new equals the cached value: no change
    _, _, r2b = gamma.block_pass(xin, codecs.f32_to_bf16(2 * prev), prev, computed=True, cache="mx")
    assert r2b == 1                                  # Delta_new = 2 x cached -> r2 = 1
    assert np.array_equal(tdc.apply(xin, prev), out)


def _tiny(steps=6, nb=2, M=40, H=64, F=128, seed=7):
    st = synthetic.stack_setup(seed, nb, H, F)
    wq = [{k: block.quantize_weights(v) for k, v in b.items()} for b in st["blocks"]]
    return st, wq, synthetic.stack_inputs(st["noise_seed"], M, H, steps)


def test_stack_without_skips_ignores_the_cache_format():
    st, wq, xs = _tiny()
    a = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.05, 0.05, 1, use_tdc=False, tdc_cache="mx")
    b = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.05, 0.05, 1, use_tdc=False)
    for x, y in zip(a["outputs"], b["outputs"]):
        assert np.array_equal(x, y)


def test_stack_skip_reuses_the_cached_value():
    st, wq, xs = _tiny()
    skips = [np.array([0, 0]), np.array([0, 0]), np.array([1, 0]), np.array([0, 0]), np.array([0, 1]),
             np.array([0, 0])]
    flags = [np.zeros(8, np.uint8)] * 6
    a = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.0, 0.0, 1, forced_flags=flags, forced_skips=skips,
                        tdc_cache="mx")
    b = block.run_stack(xs, wq, st["alpha"], st["beta"], 0.0, 0.0, 1, forced_flags=flags, forced_skips=skips)
    assert np.array_equal(a["outputs"][1], b["outputs"][1])                 # no skip yet: identical
    fa = codecs.bf16_to_f32(a["outputs"][2]).astype(np.float64)
    fb = codecs.bf16_to_f32(b["outputs"][2]).astype(np.float64)
    assert not np.array_equal(fa, fb)                                        # the skip reused a compressed Delta
    assert np.linalg.norm(fa - fb) / np.linalg.norm(fb) < 2e-2               # E4M3 keeps 3 mantissa bits
