"""Pins of the oracle's quantized linear layers: a pure-Python float64 triple
loop on tiny shapes, the unit-scale case as an exact integer matmul, and the
GELU against torch's tanh approximation."""
import math

import numpy as np
import torch

from oracle import codecs, gemm, int8, nvfp4


def _layer(seed, M, N, K):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)).astype(np.float32)
    a[:, 3] *= 12
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    bias = codecs.f32_to_bf16(rng.standard_normal(N).astype(np.float32) * 0.1)
    res = codecs.f32_to_bf16(rng.standard_normal((M, N)).astype(np.float32))
    return a, w, bias, res


def _loop_w4a4(ac, asf, ga, wc, wsf, gw, bias, gelu, res):
    A = codecs.unpack_e2m1(ac)
    W = codecs.unpack_e2m1(wc)
    M, K = A.shape
    N = W.shape[0]
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                av = float(codecs.e2m1_decode(A[m, k])) * float(codecs.e4m3_decode(asf[m, k // 16]))
                wv = float(codecs.e2m1_decode(W[n, k])) * float(codecs.e4m3_decode(wsf[n, k // 16]))
                acc += av * wv
            y = acc * float(ga) * float(gw) + float(codecs.bf16_to_f32(bias[n]))
            if gelu:
                y = 0.5 * y * (1 + math.tanh(math.sqrt(2 / math.pi) * (y + 0.044715 * y ** 3)))
            out[m, n] = y + float(codecs.bf16_to_f32(res[m, n]))
    return out


def _loop_w4a8(q, s, wc, wsf, gw, bias, gelu, res):
    W = codecs.unpack_e2m1(wc)
    M, K = q.shape
    N = W.shape[0]
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                wv = float(codecs.e2m1_decode(W[n, k])) * float(codecs.e4m3_decode(wsf[n, k // 16]))
                acc += int(q[m, k]) * wv
            y = acc * float(s[m]) * float(gw) + float(codecs.bf16_to_f32(bias[n]))
            if gelu:
                y = 0.5 * y * (1 + math.tanh(math.sqrt(2 / math.pi) * (y + 0.044715 * y ** 3)))
            out[m, n] = y + float(codecs.bf16_to_f32(res[m, n]))
    return out


def test_w4a4_matches_triple_loop():
    a, w, bias, res = _layer(0, 5, 3, 64)
    ac, asf, ga, _ = nvfp4.quantize(a)
    wc, wsf, gw, _ = nvfp4.quantize(w)
    for gelu in (False, True):
        ref = _loop_w4a4(ac, asf, ga, wc, wsf, gw, bias, gelu, res)
        got = gemm.w4a4(ac, asf, ga, wc, wsf, gw, bias=bias, gelu=gelu, residual=res, out_dtype="f32")
        assert np.allclose(got, ref, rtol=1e-6, atol=1e-6)


def test_w4a8_matches_triple_loop():
    a, w, bias, res = _layer(1, 4, 3, 48)
    q, s, _ = int8.quantize(a)
    wc, wsf, gw, _ = nvfp4.quantize(w)
    for gelu in (False, True):
        ref = _loop_w4a8(q, s, wc, wsf, gw, bias, gelu, res)
        got = gemm.w4a8(q, s, wc, wsf, gw, bias=bias, gelu=gelu, residual=res, out_dtype="f32")
        assert np.allclose(got, ref, rtol=1e-6, atol=1e-6)


def test_w4a4_no_transposed_operand():
    # a non-square case where A @ W (instead of A @ W^T) cannot even be formed
    a, w, bias, res = _layer(2, 3, 7, 32)
    ac, asf, ga, _ = nvfp4.quantize(a)
    wc, wsf, gw, _ = nvfp4.quantize(w)
    y = gemm.w4a4(ac, asf, ga, wc, wsf, gw)
    assert y.shape == (3, 7)


def test_unit_scales_give_exact_integer_matmul():
    # scale bytes 0x38 (= 1.0) and g = 1: the product is a matmul of E2M1 values,
    # i.e. (1/4) of an integer matmul of doubled values
    rng = np.random.default_rng(4)
    M, N, K = 9, 6, 64
    ac = rng.integers(0, 256, (M, K // 2)).astype(np.uint8)
    wc = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    one = np.full((M, K // 16), 0x38, np.uint8)
    onew = np.full((N, K // 16), 0x38, np.uint8)
    y = gemm.w4a4(ac, one, 1.0, wc, onew, 1.0)
    A2 = (2 * codecs.e2m1_decode(codecs.unpack_e2m1(ac))).astype(np.int64)
    W2 = (2 * codecs.e2m1_decode(codecs.unpack_e2m1(wc))).astype(np.int64)
    assert np.array_equal((4 * y.astype(np.float64)).astype(np.int64), A2 @ W2.T)
    q = rng.integers(-127, 128, (M, K)).astype(np.int8)
    y8 = gemm.w4a8(q, np.ones(M, np.float32), wc, onew, 1.0)
    assert np.array_equal((2 * y8.astype(np.float64)).astype(np.int64), q.astype(np.int64) @ W2.T)


def test_gelu_vs_torch():
    x = np.linspace(-8, 8, 2001)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(gemm.gelu_tanh(x), ref, rtol=1e-12, atol=1e-12)


def test_bf16_output_is_rounded_f32():
    a, w, bias, res = _layer(3, 4, 5, 32)
    ac, asf, ga, _ = nvfp4.quantize(a)
    wc, wsf, gw, _ = nvfp4.quantize(w)
    y32 = gemm.w4a4(ac, asf, ga, wc, wsf, gw, bias=bias, out_dtype="f32")
    y16 = gemm.w4a4(ac, asf, ga, wc, wsf, gw, bias=bias, out_dtype="bf16")
    assert np.array_equal(y16, codecs.f32_to_bf16(y32))
