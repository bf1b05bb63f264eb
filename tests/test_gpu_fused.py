"""GPU parity of the quantizing producers (quantization fused into the kernel
that produces the activation): the LayerNorm with NVFP4 / INT8 outputs and
the linear layer with an NVFP4 epilogue.

The producer's bf16 value (its y output) is compared with the oracle at the
producer's own tolerance; its codes, scale bytes, g, digit planes and row
scales must then equal the oracle's quantizers applied to that same bf16
value bit for bit (delayed scaling: NVFP4 with amax_t = headroom * the
history), and the history must hold |y|'s exact amax after every call."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import block as o_block, codecs, gemm as o_gemm, int8 as o_int8, nvfp4 as o_nvfp4
from tests.helpers import assert_gemm_close, dev, dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu


def _sb():
    import nvfp4_int8_mixed_gb300 as sb
    return sb


def _hist_words(hist):
    h = host(hist).reshape(-1).astype(np.int32)
    return h[0:1].view(np.float32)[0], int(h[1]), int(h[2])


def _set_hist(hist, amax):
    hist.zero_()
    hist[0] = int(np.array([amax], dtype=np.float32).view(np.int32)[0])


def _rows(M):
    return np.arange(M) if M <= 2048 else np.sort(np.random.default_rng(M).choice(M, 300, replace=False))


def _check_nvfp4(codes, sf, g, yf, rows, M, K, amax_t):
    rc, rsf, rg, _ = o_nvfp4.quantize(yf[rows], np.float32(amax_t))
    assert host(g)[0] == rg
    assert np.array_equal(host(codes)[rows], rc)
    got_sf = o_nvfp4.unswizzle_sf(host(sf), M, K)
    assert np.array_equal(got_sf[rows], rsf)
    Mpad = -(-M // 128) * 128
    if Mpad > M:                                     # pad rows of the swizzled layout are zero
        full = np.zeros((Mpad, K // 16), np.uint8)
        assert np.array_equal(o_nvfp4.unswizzle_sf(host(sf), Mpad, K)[M:], full[M:])


def _check_int8(planes, rs, yf, rows):
    rq, rsc, _ = o_int8.quantize(yf[rows])
    assert np.array_equal(host(rs)[rows], rsc)
    pa, pb, pc = o_int8.digit_codes(rq)
    ref = np.stack([codecs.pack_e2m1(pa), codecs.pack_e2m1(pb), codecs.pack_e2m1(pc)])
    assert np.array_equal(host(planes)[:, rows], ref)


@pytest.mark.parametrize("M,H", [(300, 256), (1, 64), (129, 1920), (17776, 1920), (5, 3072),
                                 # enough rows that every warp of the row-prefetch forms refills its buffers:
                                 # 2 blocks a lane (8-warp CTAs), 6 and 8 blocks a lane (4-warp CTAs)
                                 (17776, 1024), (6000, 3072), (5000, 4096)])
def test_layernorm_quant_parity(M, H):
    sb = _sb()
    x = synthetic.activations(synthetic.rng(M + H), M, H, max(1, H // 100), 10.0, 50.0)
    xd = dev_bf16(x)
    u8 = dict(dtype=torch.uint8, device="cuda")
    codes = torch.full((M, H // 2), 0xAB, **u8)
    sf = torch.full((sb.sf_bytes(M, H),), 0xCD, **u8)
    g = torch.zeros(1, device="cuda")
    planes = torch.full((3, M, H // 2), 0xEF, **u8)
    rs = torch.zeros(M, device="cuda")
    y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    hist = sb.amax_history(1)[0]
    rows = _rows(M)

    # zero history: every NVFP4 code and scale is 0, g = 1; INT8 is exact
    sb.layernorm_quant(xd, y=y, nvfp4=(codes, sf, g), amax_hist=hist, int8=(planes, rs))
    yf = codecs.bf16_to_f32(host_bf16_bits(y))
    ref = codecs.bf16_to_f32(o_block.layernorm(x[rows])).astype(np.float64)
    assert np.all(np.abs(yf[rows] - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-6)
    assert not host(codes).any() and not host(sf).any() and host(g)[0] == 1.0
    amax = np.max(np.abs(yf))
    assert _hist_words(hist) == (amax, 0, 0)
    _check_int8(planes, rs, yf, rows)

    # the history now holds the exact amax: codes of the dynamic quantizer at 2 * amax
    y2 = torch.empty_like(y)
    sb.layernorm_quant(xd, y=y2, nvfp4=(codes, sf, g), amax_hist=hist)
    assert torch.equal(y, y2)
    _check_nvfp4(codes, sf, g, yf, rows, M, H, np.float32(2 * amax))
    assert _hist_words(hist) == (amax, 0, 0)

    # a history well below the true amax: the saturating path, no bf16 output
    _set_hist(hist, np.float32(0.3) * amax)
    sb.layernorm_quant(xd, nvfp4=(codes, sf, g), amax_hist=hist, headroom=1.0)
    _check_nvfp4(codes, sf, g, yf, rows, M, H, np.float32(0.3) * amax)
    assert _hist_words(hist) == (amax, 0, 0)


def test_layernorm_quant_gates():
    sb = _sb()
    M, H = 200, 512
    x = synthetic.activations(synthetic.rng(3), M, H, 5, 10.0, 50.0)
    u8 = dict(dtype=torch.uint8, device="cuda")
    codes = torch.full((M, H // 2), 0xAB, **u8)
    sf = torch.full((sb.sf_bytes(M, H),), 0xCD, **u8)
    planes = torch.full((3, M, H // 2), 0xEF, **u8)
    rs = torch.full((M,), 5.0, device="cuda")
    g = torch.full((1,), 7.0, device="cuda")
    zero, one = torch.zeros(1, **u8), torch.ones(1, **u8)
    hist = sb.amax_history(1)[0]
    y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    sb.layernorm_quant(dev_bf16(x), y=y, nvfp4=(codes, sf, g), amax_hist=hist, nv_pred=zero, int8=(planes, rs),
                       i8_pred=zero)
    assert (host(codes) == 0xAB).all() and (host(sf) == 0xCD).all() and host(g)[0] == 7.0
    assert (host(planes) == 0xEF).all() and (host(rs) == 5.0).all()
    amax = np.max(np.abs(codecs.bf16_to_f32(host_bf16_bits(y))))
    assert _hist_words(hist)[0] == amax                # the history is kept whatever the gates say
    # the whole call gated off: nothing changes, the history included
    _set_hist(hist, 1.5)
    sb.layernorm_quant(dev_bf16(x), y=y, nvfp4=(codes, sf, g), amax_hist=hist, pred=zero)
    assert _hist_words(hist) == (np.float32(1.5), 0, 0) and (host(codes) == 0xAB).all()
    sb.layernorm_quant(dev_bf16(x), nvfp4=(codes, sf, g), amax_hist=hist, nv_pred=one, int8=(planes, rs),
                       i8_pred=zero)
    assert not (host(codes) == 0xAB).all() and (host(planes) == 0xEF).all()


def _operands(seed, mode, M, N, K):
    g = synthetic.rng(seed)
    a = synthetic.activations(g, M, K, max(1, K // 100), 10.0, 50.0)
    w = synthetic.weights(g, N, K)
    bias = synthetic.bias(g, N)
    wc, wsf, gw, _ = o_nvfp4.quantize(w)
    dw = (dev(wc), dev(o_nvfp4.swizzle_sf(wsf)), torch.tensor([gw], device="cuda"))
    af = codecs.bf16_to_f32(a)
    if mode == "w4a4":
        ac, asf, ga, _ = o_nvfp4.quantize(af)
        ref_fn = lambda rows, **kw: o_gemm.w4a4(ac[rows], asf[rows], ga, wc, wsf, gw, **kw)
        dev_a = dict(a=dev(ac), a_sf=dev(o_nvfp4.swizzle_sf(asf)), g_a=torch.tensor([ga], device="cuda"))
    else:
        q, s, _ = o_int8.quantize(af)
        pa, pb, pc = o_int8.digit_codes(q)
        planes = np.stack([codecs.pack_e2m1(pa), codecs.pack_e2m1(pb), codecs.pack_e2m1(pc)])
        ref_fn = lambda rows, **kw: o_gemm.w4a8(q[rows], s[rows], wc, wsf, gw, **kw)
        dev_a = dict(a=dev(planes), row_scale=dev(s))
    return dev_a, dw, bias, ref_fn


QOUT_CASES = [
    # mode, M, N, K, gelu, bias
    ("w4a4", 256, 512, 256, True, True),
    ("w4a8", 200, 192, 320, True, False),
    ("w4a4", 1, 128, 64, False, False),
    ("w4a8", 129, 256, 1920, False, True),
    ("w4a4", 300, 384, 256, True, True),                # half-width last column tiles
    ("w4a8", 300, 320, 448, False, True),
    ("w4a4", 17776, 7680, 1920, True, False),          # the FFN up-projection of the 2B block
    ("w4a8", 17776, 7680, 1920, True, False),
]


@pytest.mark.parametrize("mode,M,N,K,gelu,use_bias", QOUT_CASES)
def test_qlinear_qout_parity(mode, M, N, K, gelu, use_bias):
    sb = _sb()
    dev_a, dw, bias, ref_fn = _operands(M + N + K, mode, M, N, K)
    u8 = dict(dtype=torch.uint8, device="cuda")
    codes = torch.full((M, N // 2), 0xAB, **u8)
    sf = torch.full((sb.sf_bytes(M, N),), 0xCD, **u8)
    g = torch.full((1,), 7.0, device="cuda")
    hist = sb.amax_history(1)[0]
    zero, one = torch.zeros(1, **u8), torch.ones(1, **u8)
    kw = dict(bias=dev_bf16(bias) if use_bias else None, gelu=gelu)
    rows = _rows(M)

    # gate 0: the bf16 result is written (an INT8 next layer) and the history records its amax
    y = sb.qlinear_qout(mode, dev_a["a"], *dw, codes, sf, g, hist, a_sf=dev_a.get("a_sf"), g_a=dev_a.get("g_a"),
                        row_scale=dev_a.get("row_scale"), q_pred=zero, **kw)
    yf = codecs.bf16_to_f32(host_bf16_bits(y))
    ref = ref_fn(rows, bias=bias if use_bias else None, gelu=gelu, out_dtype="bf16")
    assert_gemm_close(yf[rows], codecs.bf16_to_f32(ref), "bf16")
    assert (host(codes) == 0xAB).all() and (host(sf) == 0xCD).all() and host(g)[0] == 7.0
    amax = np.max(np.abs(yf))
    assert _hist_words(hist) == (amax, 0, 0)

    # gate 1: NVFP4 codes of that same bf16 result, delayed scale 2 * amax; y untouched
    y2 = torch.full_like(y, 3.0)
    sb.qlinear_qout(mode, dev_a["a"], *dw, codes, sf, g, hist, a_sf=dev_a.get("a_sf"), g_a=dev_a.get("g_a"),
                    row_scale=dev_a.get("row_scale"), q_pred=one, y=y2, **kw)
    assert (y2 == 3.0).all()
    _check_nvfp4(codes, sf, g, yf, rows, M, N, np.float32(2 * amax))
    assert _hist_words(hist) == (amax, 0, 0)

    # no gate, headroom 1, a history below the amax: the saturating path
    _set_hist(hist, np.float32(0.5) * amax)
    sb.qlinear_qout(mode, dev_a["a"], *dw, codes, sf, g, hist, a_sf=dev_a.get("a_sf"), g_a=dev_a.get("g_a"),
                    row_scale=dev_a.get("row_scale"), headroom=1.0, y=y2, **kw)
    _check_nvfp4(codes, sf, g, yf, rows, M, N, np.float32(0.5) * amax)
    assert _hist_words(hist) == (amax, 0, 0)


def test_qout_feeds_the_next_layer():
    """LN -> NVFP4 (fused) -> W4A4 with a quantizing GELU epilogue -> W4A4 consumer
    equals the oracle chain on the same history values."""
    sb = _sb()
    M, H, F = 300, 256, 512
    st = synthetic.stack_setup(9, 1, H, F)
    x = synthetic.stack_inputs(st["noise_seed"], M, H, 1)[0]
    wq = {k: sb.quantize_weight_nvfp4(torch.as_tensor(st["blocks"][0][k]).cuda()) for k in ("up", "down")}
    u8 = dict(dtype=torch.uint8, device="cuda")
    c1, s1, g1 = torch.empty((M, H // 2), **u8), torch.empty(sb.sf_bytes(M, H), **u8), torch.empty(1, device="cuda")
    c2, s2, g2 = torch.empty((M, F // 2), **u8), torch.empty(sb.sf_bytes(M, F), **u8), torch.empty(1, device="cuda")
    hist = sb.amax_history(2)
    h = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    u = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):                               # second pass: both histories hold the exact amaxes
        sb.layernorm_quant(dev_bf16(x), y=h, nvfp4=(c1, s1, g1), amax_hist=hist[0])
        sb.qlinear_qout("w4a4", c1, *wq["up"], c2, s2, g2, hist[1], a_sf=s1, g_a=g1, gelu=True, y=u,
                        q_pred=torch.zeros(1, **u8))
    sb.layernorm_quant(dev_bf16(x), y=h, nvfp4=(c1, s1, g1), amax_hist=hist[0])
    sb.qlinear_qout("w4a4", c1, *wq["up"], c2, s2, g2, hist[1], a_sf=s1, g_a=g1, gelu=True)
    out = sb.qlinear_w4a4(c2, s2, g2, *wq["down"], out_dtype=torch.float32)
    # oracle: the dynamic chain (power-of-two headroom, unchanged amaxes)
    rw = {k: o_block.quantize_weights(st["blocks"][0][k]) for k in ("up", "down")}
    hf = codecs.bf16_to_f32(host_bf16_bits(h))
    hc, hsf, hg, _ = o_nvfp4.quantize(hf)
    ref_u = o_gemm.w4a4(hc, hsf, hg, rw["up"]["codes"], rw["up"]["sf"], rw["up"]["g"], gelu=True, out_dtype="bf16")
    uf = codecs.bf16_to_f32(host_bf16_bits(u))
    assert_gemm_close(uf, codecs.bf16_to_f32(ref_u), "bf16")
    rc, rsf, rg, _ = o_nvfp4.quantize(uf)
    ref = o_gemm.w4a4(rc, rsf, rg, rw["down"]["codes"], rw["down"]["sf"], rw["down"]["g"])
    assert_gemm_close(host(out), ref, "f32")


@pytest.mark.parametrize("mode,M,N,K", [("w4a4", 300, 512, 256), ("w4a8", 129, 144, 320), ("w4a8", 260, 384, 256),
                                        ("w4a4", 17776, 7680, 1920)])
def test_qlinear_amax_side_output(mode, M, N, K):
    """No NVFP4 outputs: the plain layer (bit-identical y) plus the exact
    max |y| in the history's first word, usable as a quantizer's amax_in."""
    sb = _sb()
    dev_a, dw, bias, ref_fn = _operands(M * 3 + N + K, mode, M, N, K)
    hist = sb.amax_history(1)[0]
    y = sb.qlinear_qout(mode, dev_a["a"], *dw, None, None, None, hist, a_sf=dev_a.get("a_sf"), g_a=dev_a.get("g_a"),
                        row_scale=dev_a.get("row_scale"), gelu=True, bias=dev_bf16(bias))
    if mode == "w4a4":
        y_plain = sb.qlinear_w4a4(dev_a["a"], dev_a["a_sf"], dev_a["g_a"], *dw, bias=dev_bf16(bias), gelu=True)
    else:
        y_plain = sb.qlinear_w4a8(dev_a["a"], dev_a["row_scale"], *dw, bias=dev_bf16(bias), gelu=True)
    assert torch.equal(y, y_plain)
    yf = codecs.bf16_to_f32(host_bf16_bits(y))
    assert _hist_words(hist) == (np.max(np.abs(yf)), 0, 0)
    assert host(sb.amax_hist_value(hist))[0] == np.max(np.abs(yf))
    if N % 64:
        return                                            # NVFP4 needs K % 64 == 0 for the next layer
    # the amax as a quantizer's input: the same codes as the quantizer's own amax pass
    c1, s1, g1 = sb.quantize_act_nvfp4(y, amax_in=sb.amax_hist_value(hist))
    c2, s2, g2 = sb.quantize_act_nvfp4(y)
    assert torch.equal(c1, c2) and torch.equal(s1, s2) and torch.equal(g1, g2)


def test_empty_and_zero_inputs():
    """M = 0: nothing launches and the history is left alone.  An all-zero
    input has a LayerNorm output of zeros: zero codes and scales, a zero
    amax recorded, and an INT8 row scale of 0."""
    sb = _sb()
    u8 = dict(dtype=torch.uint8, device="cuda")
    hist = sb.amax_history(1)[0]
    _set_hist(hist, 2.5)
    # zero-row views of real buffers (an empty allocation may have a null pointer, which the ABI rejects)
    x0 = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")[:0]
    c0, s0 = torch.zeros((4, 128), **u8), torch.zeros(sb.sf_bytes(4, 256), **u8)
    sb.layernorm_quant(x0, nvfp4=(c0[:0], s0, torch.empty(1, device="cuda")), amax_hist=hist)
    w = synthetic.weights(synthetic.rng(1), 128, 256)
    wq = sb.quantize_weight_nvfp4(torch.from_numpy(w).cuda())
    y0 = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")[:0]
    sb.qlinear_qout("w4a4", c0[:0], *wq, None, None, None, hist, a_sf=s0, g_a=torch.ones(1, device="cuda"), y=y0)
    assert _hist_words(hist) == (np.float32(2.5), 0, 0)
    M, H = 130, 256
    z = torch.zeros((M, H), dtype=torch.bfloat16, device="cuda")
    codes = torch.full((M, H // 2), 0xAB, **u8)
    sf = torch.full((sb.sf_bytes(M, H),), 0xCD, **u8)
    planes = torch.full((3, M, H // 2), 0xEF, **u8)
    rs = torch.full((M,), 7.0, device="cuda")
    sb.layernorm_quant(z, nvfp4=(codes, sf, torch.empty(1, device="cuda")), amax_hist=hist, int8=(planes, rs))
    assert not host(codes).any() and not host(sf).any() and not host(planes).any() and not host(rs).any()
    assert _hist_words(hist) == (np.float32(0.0), 0, 0)
