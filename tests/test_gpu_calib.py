"""GPU parity of the DMPQ calibration side: the pair-statistics reduction
(bit-exact against the oracle's fixed tree), and the calibration driver's layer errors
and fitted lines against the oracle."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import calib as o_calib, codecs, gemm as o_gemm, int8 as o_int8, nvfp4 as o_nvfp4
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
    assert np.array_equal(got, o_calib.pair_sums_tree(ah, bh)), (got, o_calib.pair_sums_tree(ah, bh))
    assert np.allclose(got, o_calib.pair_sums(ah, bh), rtol=1e-5, atol=0)


def test_calibration_lines_tiny_stack():
    from nvfp4_int8_mixed_gb300.calibration import calibrate_lines
    from nvfp4_int8_mixed_gb300.stack import DiTStack
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
    # step 0, block 0, QKV: the oracle's E_rel of the device's own layer input
    # (captured from an eager replay of step 0; the run is deterministic)
    cap = {}
    stack.tau, stack.max_skip = float("-inf"), 0
    stack.reset()
    stack.x_in.copy_(xs_dev[0])
    stack.step_dev.fill_(0)
    stack.enqueue_step(hook=lambda l, i, x: cap.setdefault((l, i), x.clone()))
    torch.cuda.synchronize()
    from tests.helpers import host_bf16_bits
    for (l, i), name in (((0, 0), "qkv"), ((1, 3), "down")):
        h = host_bf16_bits(cap[(l, i)])
        w = np.asarray(st["blocks"][l][name], np.float32)
        y_ref = codecs.bf16_to_f32(h).astype(np.float64) @ w.astype(np.float64).T
        wc, wsf, gw, _ = o_nvfp4.quantize(w)
        ac, asf, ga, _ = o_nvfp4.quantize(codecs.bf16_to_f32(h))
        y4 = o_gemm.w4a4(ac, asf, ga, wc, wsf, gw, out_dtype="f32")
        q, rs, _ = o_int8.quantize(codecs.bf16_to_f32(h))
        y8 = o_gemm.w4a8(q, rs, wc, wsf, gw, out_dtype="f32")
        k = 4 * l + i
        assert e4[0, k] == pytest.approx(o_calib.rel_l2(y4, y_ref), rel=1e-4)
        assert e8[0, k] == pytest.approx(o_calib.rel_l2(y8, y_ref), rel=1e-4)
