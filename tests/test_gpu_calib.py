"""GPU parity of the DMPQ calibration side: the pair-statistics reduction
against the oracle's float64 sums, and the calibration driver's layer errors
and fitted lines against the oracle."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import block as o_block, calib as o_calib, codecs, gemm as o_gemm, nvfp4 as o_nvfp4
from tests.helpers import dev, dev_bf16, host

pytestmark = pytest.mark.gpu


def _sb():
    import nvfp4_int8_mixed_gb300 as sb
    return sb


@pytest.mark.parametrize("n,ta,tb", [(8, "bf16", "bf16"), (8192 * 3 + 40, "bf16", "f32"), (100000, "f32", "bf16"),
                                     (1 << 20, "f32", "f32"), (17776 * 1920, "bf16", "bf16")])
def test_pair_stats_parity(n, ta, tb):
    sb = _sb()
    rng = np.random.default_rng(n)
    b = rng.standard_normal(n).astype(np.float32)
    a = (b + 0.1 * rng.standard_normal(n)).astype(np.float32)
    to = lambda v, t: dev_bf16(codecs.f32_to_bf16(v)) if t == "bf16" else dev(v)
    ad, bd = to(a, ta), to(b, tb)
    got = host(sb.pair_stats(ad, bd))
    ah = codecs.bf16_to_f32(codecs.f32_to_bf16(a)) if ta == "bf16" else a
    bh = codecs.bf16_to_f32(codecs.f32_to_bf16(b)) if tb == "bf16" else b
    ref = o_calib.pair_sums(ah, bh)
    assert np.allclose(got, ref, rtol=1e-4, atol=0), (got, ref)
    assert np.array_equal(host(sb.pair_stats(ad, bd)), got)        # fixed reduction order


def test_calibration_lines_tiny_stack():
    from nvfp4_int8_mixed_gb300.stack import DiTStack, calibrate_lines
    nb, M, H, F, T = 2, 300, 256, 512, 5
    st = synthetic.stack_setup(11, nb, H, F)
    xs = synthetic.stack_inputs(st["noise_seed"], M, H, T)
    xs_dev = [dev_bf16(x) for x in xs]
    stack = DiTStack(st["blocks"], st["alpha"], st["beta"], M, H, F, tau=0.0)
    r = calibrate_lines(stack, xs_dev, st["blocks"])
    e4, e8, gam = r["e_rel_nvfp4"], r["e_rel_int8"], r["gamma"]
    assert e4.shape == (T, 4 * nb) and np.isfinite(e4).all() and np.isfinite(e8).all()
    assert (e8 < e4).all() and (e4 < 0.5).all()                  # INT8 activations: the smaller error
    # the fitted lines are the least-squares fit of the measured series
    lb = np.repeat(np.arange(nb), 4)
    for k in range(4 * nb):
        a, b = o_calib.fit_line(gam[:T - 1, lb[k]], e4[1:, k])
        assert r["alpha"][k] == pytest.approx(a, rel=1e-9, abs=1e-12)
        assert r["beta"][k] == pytest.approx(b, rel=1e-9, abs=1e-12)
    assert np.isnan(r["delta_cos"][0]).all()
    c = r["delta_cos"][1:]
    assert (c <= 1.0 + 1e-9).all() and (c >= -1.0 - 1e-9).all() and (r["delta_rel"][1:] >= 0).all()
    # step 0, block 0, QKV: the layer input is LN(x_0); recompute its E_rel in the oracle
    h1 = o_block.layernorm(xs[0])
    w = np.asarray(st["blocks"][0]["qkv"], np.float32)
    y_ref = codecs.bf16_to_f32(h1).astype(np.float64) @ w.astype(np.float64).T
    wc, wsf, gw, _ = o_nvfp4.quantize(w)
    ac, asf, ga, _ = o_nvfp4.quantize(codecs.bf16_to_f32(h1))
    y4 = o_gemm.w4a4(ac, asf, ga, wc, wsf, gw, out_dtype="f32")
    assert e4[0, 0] == pytest.approx(o_calib.rel_l2(y4, y_ref), rel=2e-2)
