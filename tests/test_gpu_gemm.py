"""GPU parity of the W4A4 and W4A8 linear layers (a5, a6) against the
oracle's float64 product of the same quantized operands: max relative error
1e-3 on fp32 outputs (plus one bf16 rounding for bf16 outputs)."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import codecs, gemm as o_gemm, int8 as o_int8, nvfp4 as o_nvfp4
from tests.helpers import assert_gemm_close, dev, dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu


def _sb():
    import nvfp4_int8_mixed_gb300 as sb
    return sb


def _operands(seed, M, N, K, outliers=True):
    g = synthetic.rng(seed)
    a = synthetic.activations(g, M, K, max(1, K // 100) if outliers else 0, 10.0, 50.0)
    w = synthetic.weights(g, N, K)
    bias = synthetic.bias(g, N)
    res = codecs.f32_to_bf16(g.standard_normal((M, N), dtype=np.float32))
    return a, w, bias, res


def _oracle_w(w):
    wc, wsf, gw, _ = o_nvfp4.quantize(w)
    return wc, wsf, gw


def _dev_w(wc, wsf, gw):
    return dev(wc), dev(o_nvfp4.swizzle_sf(wsf)), torch.tensor([gw], device="cuda")


CASES = [
    # M, N, K, gelu, bias, residual, out
    (256, 512, 256, False, False, False, "f32"),      # config-1 layer
    (256, 512, 256, True, True, True, "bf16"),
    (200, 144, 320, False, True, False, "f32"),       # ragged M, N tail (144 = 128 + 16), K tail (320 = 256 + 64)
    (129, 256, 1920, True, False, True, "bf16"),      # K = 1920: half a K step at the end
    (1, 128, 64, False, False, False, "f32"),
    (384, 384, 7680, False, True, True, "f32"),
    # a ragged last column of <= 128 columns runs as half-width tiles after all full tiles
    (300, 320, 448, True, True, True, "bf16"),       # 64 valid columns: one CTA's W half lies wholly past N
    (520, 1920, 256, False, True, True, "bf16"),     # 7 full column tiles + 1 half, 3 row tiles
    (600, 5760, 128, False, False, False, "f32"),    # the QKV width: 22 full column tiles + 1 half
]


@pytest.mark.parametrize("M,N,K,gelu,use_bias,use_res,out", CASES)
def test_w4a4_parity(M, N, K, gelu, use_bias, use_res, out):
    sb = _sb()
    a, w, bias, res = _operands(M + N + K, M, N, K)
    ac, asf, ga, _ = o_nvfp4.quantize(codecs.bf16_to_f32(a))
    wc, wsf, gw = _oracle_w(w)
    ref = o_gemm.w4a4(ac, asf, ga, wc, wsf, gw, bias=bias if use_bias else None, gelu=gelu,
                      residual=res if use_res else None, out_dtype=out)
    dw = _dev_w(wc, wsf, gw)
    y = sb.qlinear_w4a4(dev(ac), dev(o_nvfp4.swizzle_sf(asf)), torch.tensor([ga], device="cuda"), *dw,
                        bias=dev_bf16(bias) if use_bias else None, residual=dev_bf16(res) if use_res else None,
                        gelu=gelu, out_dtype=torch.float32 if out == "f32" else torch.bfloat16)
    sb.get_error()
    got = host(y) if out == "f32" else codecs.bf16_to_f32(host_bf16_bits(y))
    refv = ref if out == "f32" else codecs.bf16_to_f32(ref)
    assert_gemm_close(got, refv, out)


@pytest.mark.parametrize("M,N,K,gelu,use_bias,use_res,out", CASES)
def test_w4a8_parity(M, N, K, gelu, use_bias, use_res, out):
    sb = _sb()
    a, w, bias, res = _operands(M + N + K + 1, M, N, K)
    q, s, _ = o_int8.quantize(codecs.bf16_to_f32(a))
    pa, pb, pc = o_int8.digit_codes(q)
    planes = np.stack([codecs.pack_e2m1(pa), codecs.pack_e2m1(pb), codecs.pack_e2m1(pc)])
    wc, wsf, gw = _oracle_w(w)
    ref = o_gemm.w4a8(q, s, wc, wsf, gw, bias=bias if use_bias else None, gelu=gelu,
                      residual=res if use_res else None, out_dtype=out)
    y = sb.qlinear_w4a8(dev(planes), dev(s), *_dev_w(wc, wsf, gw),
                        bias=dev_bf16(bias) if use_bias else None, residual=dev_bf16(res) if use_res else None,
                        gelu=gelu, out_dtype=torch.float32 if out == "f32" else torch.bfloat16)
    sb.get_error()
    got = host(y) if out == "f32" else codecs.bf16_to_f32(host_bf16_bits(y))
    refv = ref if out == "f32" else codecs.bf16_to_f32(ref)
    assert_gemm_close(got, refv, out)


def test_unit_scale_exact_integer_products():
    """All scales 1 (E4M3 0x38) and g = 1: each output is (1/4) x an integer
    sum small enough for fp32 -- the kernel must be exact."""
    sb = _sb()
    rng = np.random.default_rng(0)
    M, N, K = 256, 256, 512
    ac = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    wc = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    ones_a = np.full((M, K // 16), 0x38, np.uint8)
    ones_w = np.full((N, K // 16), 0x38, np.uint8)
    ref = o_gemm.w4a4(ac, ones_a, 1.0, wc, ones_w, 1.0)
    one = torch.ones(1, device="cuda")
    y = sb.qlinear_w4a4(dev(ac), dev(o_nvfp4.swizzle_sf(ones_a)), one, dev(wc), dev(o_nvfp4.swizzle_sf(ones_w)), one,
                        out_dtype=torch.float32)
    assert np.array_equal(host(y), ref)


def test_quantize_then_gemm_chain():
    """GPU quantizers feeding the GPU GEMMs == oracle quantizers feeding the oracle GEMMs."""
    sb = _sb()
    M, N, K = 300, 256, 1920
    a, w, bias, res = _operands(5, M, N, K)
    x = dev_bf16(a)
    wc, wsf, gw = sb.quantize_weight_nvfp4(dev(w))
    codes, sf, ga = sb.quantize_act_nvfp4(x)
    y4 = sb.qlinear_w4a4(codes, sf, ga, wc, wsf, gw, out_dtype=torch.float32)
    _, planes, s = sb.quantize_act_int8(x, want_q=False)
    y8 = sb.qlinear_w4a8(planes, s, wc, wsf, gw, out_dtype=torch.float32)
    rwc, rwsf, rgw = _oracle_w(w)
    rac, rasf, rga, _ = o_nvfp4.quantize(codecs.bf16_to_f32(a))
    rq, rs, _ = o_int8.quantize(codecs.bf16_to_f32(a))
    assert_gemm_close(host(y4), o_gemm.w4a4(rac, rasf, rga, rwc, rwsf, rgw), "f32")
    assert_gemm_close(host(y8), o_gemm.w4a8(rq, rs, rwc, rwsf, rgw), "f32")


def test_pred_zero_skips_gemm():
    sb = _sb()
    M, N, K = 128, 128, 256
    a, w, _, _ = _operands(6, M, N, K)
    ac, asf, ga, _ = o_nvfp4.quantize(codecs.bf16_to_f32(a))
    wc, wsf, gw = _oracle_w(w)
    y = torch.full((M, N), 5.0, device="cuda")
    pred = torch.zeros(1, dtype=torch.uint8, device="cuda")
    sb.qlinear_w4a4(dev(ac), dev(o_nvfp4.swizzle_sf(asf)), torch.tensor([ga], device="cuda"), *_dev_w(wc, wsf, gw),
                    out=y, pred=pred)
    assert (host(y) == 5.0).all()


@pytest.mark.parametrize("name,K,N,gelu,use_res", synthetic.GEMM_SHAPES["2B"])
def test_2b_shapes_sampled_rows(name, K, N, gelu, use_res):
    """Config-2 shapes at full size in the bench's launch configuration; the
    oracle checks a sample of rows (all N columns)."""
    _full_shape_sampled_rows(K, N, gelu, use_res)


@pytest.mark.parametrize("name,K,N,gelu,use_res", synthetic.GEMM_SHAPES["5B"])
def test_5b_shapes_sampled_rows(name, K, N, gelu, use_res):
    """Config-3 shapes (5B-class set, M=17776, K 3072/12288, N up to 12288) at
    full size; the oracle checks a sample of rows (all N columns)."""
    _full_shape_sampled_rows(K, N, gelu, use_res)


def _full_shape_sampled_rows(K, N, gelu, use_res):
    sb = _sb()
    M = synthetic.M_2B
    lay = synthetic.gemm_layer(1, M, K, N, use_res)
    a, w = lay["a"], lay["w"]
    x = dev_bf16(a)
    wc, wsf, gw = sb.quantize_weight_nvfp4(dev(w))
    res = dev_bf16(lay["residual"]) if use_res else None
    codes, sf, ga = sb.quantize_act_nvfp4(x)
    y4 = sb.qlinear_w4a4(codes, sf, ga, wc, wsf, gw, residual=res, gelu=gelu)
    _, planes, s = sb.quantize_act_int8(x, want_q=False)
    y8 = sb.qlinear_w4a8(planes, s, wc, wsf, gw, residual=res, gelu=gelu)
    sb.get_error()
    rows = np.r_[0:2, M - 2:M, np.random.default_rng(K + N).choice(M, 28, replace=False)]
    af = codecs.bf16_to_f32(a)
    amax_t = np.float32(np.max(np.abs(af)))
    rwc, rwsf, rgw = _oracle_w(w)
    rac, rasf, rga, _ = o_nvfp4.quantize(af[rows], amax_t)
    rr = lay["residual"][rows] if use_res else None
    ref4 = o_gemm.w4a4(rac, rasf, rga, rwc, rwsf, rgw, gelu=gelu, residual=rr, out_dtype="bf16")
    rq, rs, _ = o_int8.quantize(af[rows])
    ref8 = o_gemm.w4a8(rq, rs, rwc, rwsf, rgw, gelu=gelu, residual=rr, out_dtype="bf16")
    assert_gemm_close(codecs.bf16_to_f32(host_bf16_bits(y4)[rows]), codecs.bf16_to_f32(ref4), "bf16")
    assert_gemm_close(codecs.bf16_to_f32(host_bf16_bits(y8)[rows]), codecs.bf16_to_f32(ref8), "bf16")
