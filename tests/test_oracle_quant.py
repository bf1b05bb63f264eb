"""Pins of the oracle's NVFP4 and INT8 quantizers: hand-built blocks with
known scales, closed-form cases, brute-force nearest codes, the scale-factor
layout's fixed points, INT8 corner cases and the digit split."""
import numpy as np
import pytest

from oracle import codecs, int8, nvfp4

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)


def _q(x, amax=None):
    return nvfp4.quantize(np.asarray(x, dtype=np.float32), amax)


def test_block_at_tensor_amax_gets_max_scale():
    x = np.zeros((1, 32), np.float32)
    x[0, :16] = np.linspace(-3, 3, 16)
    x[0, 5] = -7.0                            # tensor amax, in block 0
    x[0, 16:] = 0.5
    codes, sf, g, amax = _q(x)
    assert amax == 7.0 and g == np.float32(7.0 / 2688)
    assert sf[0, 0] == 0x7E                   # S = 448
    c = codecs.unpack_e2m1(codes)[0]
    assert c[5] == 0xF                        # -6: the block maximum maps to the top code


def test_known_scales_recover_grid_exactly():
    # amax_t = 2688 -> g = 1, so s = amax_b / 6; blocks built as S * grid values
    rng = np.random.default_rng(0)
    for S in [448.0, 1.0, 0.5, 3.5, 40.0, 2.0 ** -6, 2.0 ** -8]:
        vals = rng.choice(np.concatenate([GRID, -GRID]), 16).astype(np.float32)
        vals[3] = 6.0                         # block max = 6 S
        x = np.zeros((1, 32), np.float32)
        x[0, :16] = vals * np.float32(S)
        x[0, 16] = 2688.0                     # second block carries the tensor amax
        codes, sf, g, _ = _q(x)
        assert g == 1.0
        assert codecs.e4m3_decode(sf[0, 0]) == np.float32(S)
        deq = nvfp4.dequantize(codes, sf, g)[0, :16]
        assert np.array_equal(deq, (vals * np.float32(S)).astype(np.float64))


def test_zero_block_and_zero_tensor():
    x = np.zeros((2, 32), np.float32)
    x[1, 20] = 1.0
    codes, sf, g, _ = _q(x)
    assert sf[0, 0] == 0 and sf[0, 1] == 0 and sf[1, 0] == 0
    assert not codes[0].any()
    codes, sf, g, amax = _q(np.zeros((3, 16), np.float32))
    assert amax == 0 and g == 1.0 and not sf.any() and not codes.any()


def test_tiny_block_gets_subnormal_scale_or_zero():
    x = np.zeros((1, 48), np.float32)
    x[0, 0] = 448.0                           # amax_t; g = 1/6
    x[0, 16] = 6.0 * 2.0 ** -9 / 6 * 6        # amax_b = 6 * 2^-9 -> s = amax_b*448/448 = 6*2^-9 -> S code 0x06
    x[0, 32] = 2.0 ** -12                     # s = 2^-12 < half of min subnormal -> S = 0, codes +0
    x[0, 33] = -2.0 ** -13
    codes, sf, g, _ = _q(x)
    assert sf[0, 1] == 0x06
    assert sf[0, 2] == 0
    c = codecs.unpack_e2m1(codes)[0]
    assert c[32] == 0 and c[33] == 0          # +0 for a block whose scale is zero


def test_codes_are_nearest_brute_force():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((8, 64)).astype(np.float32) * 3
    x[:, 7] *= 20
    codes, sf, g, amax = _q(x)
    c = codecs.unpack_e2m1(codes)
    S = codecs.e4m3_decode(sf).astype(np.float32)
    for i in range(8):
        for k in range(64):
            d = np.float32(S[i, k // 16] * g)
            if d == 0:
                assert c[i, k] == 0
                continue
            v = np.float32(x[i, k] * np.float32(np.float32(1.0) / d))
            a = min(abs(float(v)), 6.0)
            dist = np.abs(GRID.astype(np.float64) - a)
            best = np.flatnonzero(dist == dist.min())
            expect = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
            assert (c[i, k] & 7) == expect and (c[i, k] >> 3) == int(np.signbit(v))


def test_caller_amax_below_true_amax_saturates():
    x = np.full((1, 16), 10.0, np.float32)
    codes, sf, g, _ = _q(x, amax=np.float32(5.0))
    assert sf[0, 0] == 0x7E                  # s = 896 clamps to 448
    assert (codecs.unpack_e2m1(codes)[0] == 7).all()


def test_relative_error_bound():
    # with the E4M3 scale rounding, the block max still maps within the E2M1 range,
    # and each element's error is at most half a grid step at the element's scale
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    codes, sf, g, _ = _q(x)
    deq = nvfp4.dequantize(codes, sf, g)
    S = codecs.e4m3_decode(sf).astype(np.float64) * float(g)
    err = np.abs(deq - x).reshape(64, 16, 16)
    # largest E2M1 step is 2 (between 4 and 6) -> half-step 1 * d; beyond 6*d saturation error
    lim = np.maximum(1.0 * S, np.abs(x).reshape(64, 16, 16).max(axis=2) - 6 * S)[:, :, None]
    assert (err <= lim + 1e-12).all()


def test_sf_layout_fixed_points_and_bijection():
    kc4 = 8
    off = lambda m, c: int(nvfp4.sf_offset(m, c, kc4))
    assert off(0, 0) == 0 and off(1, 0) == 16 and off(31, 0) == 31 * 16
    assert off(32, 0) == 4 and off(96, 0) == 12 and off(0, 1) == 1 and off(0, 3) == 3
    assert off(0, 4) == 512 and off(128, 0) == 512 * (kc4 // 4)
    R, K = 200, 128
    rp, kc = nvfp4.sf_padded_shape(R, K)
    m, c = np.meshgrid(np.arange(rp), np.arange(kc), indexing="ij")
    offs = nvfp4.sf_offset(m, c, kc).ravel()
    assert np.array_equal(np.sort(offs), np.arange(rp * kc))
    sf = np.random.default_rng(0).integers(1, 255, (R, K // 16)).astype(np.uint8)
    buf = nvfp4.swizzle_sf(sf)
    assert buf.size == rp * kc and np.array_equal(nvfp4.unswizzle_sf(buf, R, K), sf)
    assert buf.astype(np.int64).sum() == sf.astype(np.int64).sum()   # pads are zero


# ------------------------------------------------------------------ INT8
def test_int8_extremes_and_zero_row():
    x = np.array([[3.0, -3.0, 1.5, 0.0], [0, 0, 0, 0], [-2.0, 1.0, 0.5, 2.0]], np.float32)
    q, s, amax = int8.quantize(x)
    assert q[0].tolist() == [127, -127, 64, 0]          # 1.5*127/3 = 63.5 -> 64 (ties to even)
    assert q[1].tolist() == [0, 0, 0, 0] and s[1] == 0
    assert q[2, 0] == -127 and q[2, 3] == 127
    assert s[0] == np.float32(3.0) / np.float32(127.0)
    assert (q != -128).all()


def test_int8_ties_to_even():
    # amax 127 -> inv = 1 exactly, so x * inv = x
    x = np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5]], np.float32)
    q, s, _ = int8.quantize(x)
    assert q[0].tolist() == [127, 2, 4, -2, 0, 0, 2]


def test_int8_saturates_with_small_caller_amax():
    x = np.array([[10.0, -10.0, 1.0]], np.float32)
    q, s, _ = int8.quantize(x, amax=np.array([2.0], np.float32))
    assert q[0].tolist() == [127, -127, 64]   # 1*63.5 -> 64


def test_digit_split_reconstructs_every_code():
    q = np.arange(-127, 128)
    a, b, c = int8.digits(q)
    assert np.array_equal(64 * a + 8 * b + c, q)
    allowed = {-4, -3, -2, -1, 0, 1, 2, 3, 4}
    assert set(a.tolist()) <= allowed and set(b.tolist()) <= allowed and set(c.tolist()) <= allowed
    ca, cb, cc = int8.digit_codes(q)
    dec = 64 * codecs.e2m1_decode(ca) + 8 * codecs.e2m1_decode(cb) + codecs.e2m1_decode(cc)
    assert np.array_equal(dec.astype(np.int64), q)
