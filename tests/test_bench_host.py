"""Host-side arithmetic of bench.py's per-GEMM roofline (no GPU): algorithmic
bytes, arithmetic intensity and the binding ceiling of each quantized linear
on the 2B-class shapes (M = 17776)."""
import pytest

M = 17776


def _bench():
    import bench
    return bench


def test_w4a4_qkv_bytes_and_intensity():
    # codes 17776*960 + scales 17776*120 + W 5760*(960+120) + bf16 y 17776*5760*2
    r = _bench().gemm_roofline("w4a4", M, 5760, 1920, False, 1e-3, 11580.0, 6785.9)
    want = M * 960 + M * 120 + 5760 * 1080 + 2 * M * 5760
    assert r["bytes"] == pytest.approx(want, rel=1e-12)
    assert r["bytes"] == pytest.approx(230.2e6, rel=1e-3)
    assert r["AI"] == pytest.approx(2 * M * 5760 * 1920 / want, rel=1e-12)
    assert round(r["AI"]) == 1708


def test_residual_doubles_the_output_bytes_and_can_make_it_hbm_bound():
    b = _bench()
    plain = b.gemm_roofline("w4a4", M, 1920, 1920, False, 1e-3, 11580.0, 6785.9)
    res = b.gemm_roofline("w4a4", M, 1920, 1920, True, 1e-3, 11580.0, 6785.9)
    assert res["bytes"] - plain["bytes"] == pytest.approx(2 * M * 1920)
    assert res["bytes"] == pytest.approx(157.8e6, rel=1e-3)
    assert round(res["AI"]) == 831
    # 6785.9 GB/s x 831 FLOP/B = 5.6 PFLOP/s, under the 11.58 PFLOP/s FP4 peak
    assert res["bound"] == "hbm"
    assert res["ceiling"] == pytest.approx(6785.9 * res["AI"] / 1e3)


def test_w4a8_reads_three_planes_and_has_a_third_of_the_fp4_ceiling():
    b = _bench()
    a4 = b.gemm_roofline("w4a4", M, 7680, 1920, False, 1e-3, 11580.0, 6785.9)
    a8 = b.gemm_roofline("w4a8", M, 7680, 1920, False, 1e-3, 11580.0, 6785.9)
    assert a8["bytes"] - a4["bytes"] == pytest.approx(3 * M * 960 + 4 * M - (M * 960 + M * 120))
    assert a8["bound"] == "tensor"
    assert a8["ceiling"] == pytest.approx(11580.0 / 3)


def test_fractions_follow_the_timed_seconds():
    b = _bench()
    flops = 2.0 * M * 7680 * 1920
    r = b.gemm_roofline("w4a8", M, 7680, 1920, False, flops / 1930e12, 11580.0, 6785.9)
    assert r["TFLOP/s"] == pytest.approx(1930.0)
    assert r["frac_tensor"] == pytest.approx(1930.0 / 3860.0)
    assert r["frac_ceiling"] == pytest.approx(r["TFLOP/s"] / r["ceiling"])
