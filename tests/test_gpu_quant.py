"""GPU parity of the quantizers (a1-a4) against the oracle: codes, scale
bytes (through the swizzled layout), tensor scales and row scales must be
bit-exact on the same seeded inputs."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import codecs, int8 as o_int8, nvfp4 as o_nvfp4
from tests.helpers import assert_gemm_close, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


def _sb():
    import nvfp4_int8_mixed_gb300 as sb
    return sb


SHAPES = [(256, 256), (1, 64), (200, 320), (129, 1920), (50, 2560), (17, 3584), (9, 5120), (300, 7680),
          (33, 10240), (5, 16384)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_nvfp4_act_bit_exact(M, K):
    sb = _sb()
    g = synthetic.rng(100 + M)
    a = synthetic.activations(g, M, K, max(1, K // 100), 10.0, 50.0)
    x = dev_bf16(a)
    codes, sf, gg = sb.quantize_act_nvfp4(x)
    rc, rsf, rg, ramax = o_nvfp4.quantize(codecs.bf16_to_f32(a))
    torch.cuda.synchronize()
    assert host(gg)[0] == rg
    assert np.array_equal(host(codes), rc)
    assert np.array_equal(host(sf), o_nvfp4.swizzle_sf(rsf))
    ta, ra = sb.amax(x, tensor=True, rows=True)
    assert host(ta)[0] == ramax
    assert np.array_equal(host(ra), o_int8.row_amax(codecs.bf16_to_f32(a)))


def test_nvfp4_caller_amax_strided_rows_and_pred():
    sb = _sb()
    g = synthetic.rng(7)
    big = synthetic.activations(g, 96, 3 * 256, 3, 20.0)
    a = np.ascontiguousarray(big[:, 512:768])           # the "V slice" of a fused QKV output
    xs = dev_bf16(big)[:, 512:768]
    amax = torch.tensor([np.float32(3.0)], device="cuda")  # below the true amax: saturation path
    codes, sf, gg = sb.quantize_act_nvfp4(xs, amax_in=amax)
    rc, rsf, rg, _ = o_nvfp4.quantize(codecs.bf16_to_f32(a), np.float32(3.0))
    assert np.array_equal(host(codes), rc) and np.array_equal(host(sf), o_nvfp4.swizzle_sf(rsf))
    assert host(gg)[0] == rg
    # pred = 0: outputs untouched
    pred = torch.zeros(1, dtype=torch.uint8, device="cuda")
    c2 = torch.full_like(codes, 0xAB)
    sf2 = torch.full_like(sf, 0xCD)
    g2 = torch.full_like(gg, 7.0)
    sb.quantize_act_nvfp4(xs, amax_in=amax, pred=pred, out=(c2, sf2, g2))
    assert (host(c2) == 0xAB).all() and (host(sf2) == 0xCD).all() and host(g2)[0] == 7.0


def test_nvfp4_all_zero_tensor():
    sb = _sb()
    x = torch.zeros((130, 128), dtype=torch.bfloat16, device="cuda")
    codes, sf, gg = sb.quantize_act_nvfp4(x)
    assert host(gg)[0] == 1.0 and not host(codes).any() and not host(sf).any()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nvfp4_weight_bit_exact(dtype):
    sb = _sb()
    w = synthetic.weights(synthetic.rng(3), 384, 1920)
    if dtype == "bf16":
        wb = codecs.f32_to_bf16(w)
        t = dev_bf16(wb)
        ref_in = codecs.bf16_to_f32(wb)
    else:
        t = dev(w)
        ref_in = w
    codes, sf, gg = sb.quantize_weight_nvfp4(t)
    rc, rsf, rg, _ = o_nvfp4.quantize(ref_in)
    assert host(gg)[0] == rg
    assert np.array_equal(host(codes), rc) and np.array_equal(host(sf), o_nvfp4.swizzle_sf(rsf))


@pytest.mark.parametrize("M,K", SHAPES)
def test_int8_bit_exact(M, K):
    sb = _sb()
    g = synthetic.rng(200 + M)
    a = synthetic.activations(g, M, K, max(1, K // 100), 10.0, 50.0)
    a[0, :] = 0                                           # a zero row
    q, planes, s = sb.quantize_act_int8(dev_bf16(a))
    rq, rs, _ = o_int8.quantize(codecs.bf16_to_f32(a))
    assert np.array_equal(host(q), rq)
    assert np.array_equal(host(s), rs)
    pa, pb, pc = o_int8.digit_codes(rq)
    ref_planes = np.stack([codecs.pack_e2m1(pa), codecs.pack_e2m1(pb), codecs.pack_e2m1(pc)])
    assert np.array_equal(host(planes), ref_planes)


def test_int8_caller_row_amax_saturates():
    sb = _sb()
    a = synthetic.activations(synthetic.rng(9), 64, 128, 2, 20.0)
    amax = np.full(64, 0.5, np.float32)
    q, planes, s = sb.quantize_act_int8(dev_bf16(a), row_amax=dev(amax))
    rq, rs, _ = o_int8.quantize(codecs.bf16_to_f32(a), amax)
    assert np.array_equal(host(q), rq) and np.array_equal(host(s), rs)


def test_quantizers_full_2b_shape_sampled_rows():
    """Config-2 activation (M=17776, K=1920 and 7680): every row through the
    kernels, a sample of rows through the oracle with the tensor amax."""
    _quantizers_full_shape(1920, 7680)


def test_quantizers_full_5b_shape_sampled_rows():
    """Config-3 activation (M=17776, K=3072 and 12288), as above."""
    _quantizers_full_shape(3072, 12288)


def _quantizers_full_shape(*Ks):
    sb = _sb()
    for K in Ks:
        lay = synthetic.gemm_layer(1, synthetic.M_2B, K, 128, False)
        a = lay["a"]
        x = dev_bf16(a)
        codes, sf, gg = sb.quantize_act_nvfp4(x)
        q, planes, s = sb.quantize_act_int8(x)
        amax_t = np.float32(np.max(np.abs(codecs.bf16_to_f32(a))))
        rows = np.r_[0:3, synthetic.M_2B - 3:synthetic.M_2B,
                     np.random.default_rng(K).choice(synthetic.M_2B, 40, replace=False)]
        rc, rsf, rg, _ = o_nvfp4.quantize(codecs.bf16_to_f32(a[rows]), amax_t)
        assert host(gg)[0] == rg
        assert np.array_equal(host(codes)[rows], rc)
        got_sf = o_nvfp4.unswizzle_sf(host(sf), synthetic.M_2B, K)[rows]
        assert np.array_equal(got_sf, rsf)
        rq, rs, _ = o_int8.quantize(codecs.bf16_to_f32(a[rows]))
        assert np.array_equal(host(q)[rows], rq) and np.array_equal(host(s)[rows], rs)
        pad = host(sf).reshape(-1)
        assert pad.size == o_nvfp4.sf_padded_shape(synthetic.M_2B, K)[0] * (K // 16)


@pytest.mark.parametrize("M,K,ldq", [(1, 64, 64), (129, 320, 320), (300, 1920, 2048)])
def test_int8_digit_planes_of_plain_codes(M, K, ldq):
    """Plain int8 codes from anywhere (here every byte value, -128 included,
    with a row stride) -> the exact digit planes; the W4A8 GEMM on them
    equals the oracle's int8 x W4 product."""
    from oracle import gemm as o_gemm
    sb = _sb()
    g = synthetic.rng(300 + M)
    full = g.integers(-128, 128, size=(M, ldq)).astype(np.int8)
    full[0, :min(K, 256)] = np.arange(-128, 128)[:min(K, 256)]           # every code value
    qd = dev(full)[:, :K]
    planes = sb.int8_digit_planes(qd)
    q = full[:, :K]
    pa, pb, pc = o_int8.digit_codes(q)
    assert np.array_equal(host(planes), np.stack([codecs.pack_e2m1(pa), codecs.pack_e2m1(pb), codecs.pack_e2m1(pc)]))
    # the W4A8 layer on planes made from plain codes
    s = g.uniform(0.001, 0.01, M).astype(np.float32)
    w = synthetic.weights(g, 128, K)
    wc, wsf, gw = sb.quantize_weight_nvfp4(dev(w))
    y = sb.qlinear_w4a8(planes, dev(s), wc, wsf, gw, out_dtype=torch.float32)
    rwc, rwsf, rgw, _ = o_nvfp4.quantize(w)
    assert_gemm_close(host(y), o_gemm.w4a8(q, s, rwc, rwsf, rgw), "f32")


def test_empty_row_count_through_the_binding():
    """M = 0 activations (an empty token batch) pass through every row call
    of the binding as no-ops with empty results, and leave the stream clean."""
    sb = _sb()
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    ta, ra = sb.amax(x, tensor=True, rows=True)
    assert ra.shape == (0,)
    codes, sf, g = sb.quantize_act_nvfp4(x)
    assert codes.shape == (0, 64) and sf.numel() == 0
    q, planes, s = sb.quantize_act_int8(x)
    assert q.shape == (0, 128) and planes.shape == (3, 0, 64) and s.shape == (0,)
    w = synthetic.rng(5).standard_normal((64, 128)).astype(np.float32) * 0.02
    wc, wsf, gw = sb.quantize_weight_nvfp4(dev(w))
    assert sb.qlinear_w4a4(codes, sf, g, wc, wsf, gw).shape == (0, 64)
    assert sb.qlinear_w4a8(planes, s, wc, wsf, gw, out_dtype=torch.float32).shape == (0, 64)
    assert sb.layernorm(x).shape == (0, 128)
    sb.get_error()
