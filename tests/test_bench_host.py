"""Host-side arithmetic of bench.py's rooflines (no GPU): algorithmic bytes,
arithmetic intensity and ceilings of each quantized linear on the 2B-class
shapes (M = 17776), the quantizers' method bytes, and the time-weighted
bound of a DiT stack run."""
import pytest

M = 17776
FP4, HBM = 11290.2, 6789.6


def _bench():
    import bench
    return bench


def test_w4a4_qkv_bytes_and_intensity():
    # codes 17776*960 + scales 17776*120 + W 5760*(960+120) + bf16 y 17776*5760*2
    r = _bench().gemm_roofline("w4a4", M, 5760, 1920, False, 1e-3, FP4, HBM)
    want = M * 960 + M * 120 + 5760 * 1080 + 2 * M * 5760
    assert r["bytes"] == pytest.approx(want, rel=1e-12) and r["bytes_moved"] == r["bytes"]
    assert r["bytes"] == pytest.approx(230.2e6, rel=1e-3)
    assert r["AI"] == pytest.approx(2 * M * 5760 * 1920 / want, rel=1e-12)
    assert round(r["AI"]) == 1708
    assert "fp4_pipe_frac" not in r


def test_residual_doubles_the_output_bytes_and_can_make_it_hbm_bound():
    b = _bench()
    plain = b.gemm_roofline("w4a4", M, 1920, 1920, False, 1e-3, FP4, HBM)
    res = b.gemm_roofline("w4a4", M, 1920, 1920, True, 1e-3, FP4, HBM)
    assert res["bytes"] - plain["bytes"] == pytest.approx(2 * M * 1920)
    assert res["bytes"] == pytest.approx(157.8e6, rel=1e-3)
    assert round(res["AI"]) == 831
    # 6789.6 GB/s x 831 FLOP/B = 5.6 PFLOP/s, under the 11.29 PFLOP/s FP4 peak
    assert res["bound"] == "hbm"
    assert res["ceiling"] == pytest.approx(HBM * res["AI"] / 1e3)


def test_w4a8_counts_int8_codes_and_reports_its_pipe_share_separately():
    b = _bench()
    a4 = b.gemm_roofline("w4a4", M, 7680, 1920, False, 1e-3, FP4, HBM)
    a8 = b.gemm_roofline("w4a8", M, 7680, 1920, False, 1e-3, FP4, HBM)
    # the method's operand: 1-byte codes and a row scale; the kernel streams three 0.5-byte digit planes
    assert a8["bytes"] - a4["bytes"] == pytest.approx(M * 1920 + 4 * M - (M * 960 + M * 120))
    assert a8["bytes_moved"] - a8["bytes"] == pytest.approx(0.5 * M * 1920)
    assert a8["ceiling"] == pytest.approx(min(FP4, HBM * a8["AI"] / 1e3))
    assert a8["design_ceiling"] == pytest.approx(FP4 / 3)


def test_fractions_follow_the_timed_seconds():
    b = _bench()
    flops = 2.0 * M * 7680 * 1920
    r = b.gemm_roofline("w4a8", M, 7680, 1920, False, flops / 1930e12, FP4, HBM)
    assert r["TFLOP/s"] == pytest.approx(1930.0)
    assert r["frac_fp4_peak"] == pytest.approx(1930.0 / FP4)            # the method's work over the FP4 peak
    assert r["fp4_pipe_frac"] == pytest.approx(3 * 1930.0 / FP4)        # three digit MMAs per product
    assert r["frac_ceiling"] == pytest.approx(r["TFLOP/s"] / r["ceiling"])


def test_quantizer_method_bytes():
    b = _bench()
    assert b.quant_bytes("nvfp4", M, 1920) == pytest.approx(2.5625 * M * 1920)
    assert b.quant_bytes("int8", M, 1920) == pytest.approx(3 * M * 1920 + 4 * M)


def test_stack_ideal_time_sums_per_kernel_bounds():
    b = _bench()
    H, F = 1920, 7680
    kinds = ("qkv", "out", "up", "down")
    zero = {k: 0 for k in kinds}
    # one skipped block: the TDC reuse and the Gamma pass, 14 B per element
    assert b.stack_ideal_seconds(M, H, F, zero, zero, 0, 1, FP4, HBM) == pytest.approx(14 * M * H / (HBM * 1e9))
    # one computed all-NVFP4 block: GEMMs at their ceilings + quantizers + LN + Gamma
    one = {k: 1 for k in kinds}
    t = b.stack_ideal_seconds(M, H, F, one, zero, 1, 0, FP4, HBM)
    want = 0.0
    for K, N, res in ((H, 3 * H, False), (H, H, True), (H, F, False), (F, H, True)):
        g = b.gemm_roofline("w4a4", M, N, K, res, 1.0, FP4, HBM)
        want += 2.0 * M * N * K / (g["ceiling"] * 1e12) + 2.5625 * M * K / (HBM * 1e9)
    want += (2 * M * H) / (HBM * 1e9)               # the V slice's amax pass
    want += (8 * M * H + 8 * M * H) / (HBM * 1e9)   # two LayerNorms + Gamma
    assert t == pytest.approx(want, rel=1e-12)
    # INT8 layers: the GEMM at a third of the FP4 peak (three digit-plane MMAs)
    t8 = b.stack_ideal_seconds(M, H, F, zero, {"qkv": 1, "out": 0, "up": 0, "down": 0}, 0, 0, FP4, HBM)
    assert t8 == pytest.approx(2.0 * M * 3 * H * H / (FP4 / 3 * 1e12) + 3 * M * H / (HBM * 1e9) + 4 * M / (HBM * 1e9))
