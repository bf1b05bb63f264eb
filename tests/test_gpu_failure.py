"""The device-error paths of the linear layers and the LayerNorm producers,
made to run on purpose.

Every mbarrier wait in the GEMM is bounded.  The test switch
sixbit_debug_stall_gemm(1) makes the MMA-issuing thread wait on a barrier
that nothing signals, so that wait gives up after its normal poll cap: the
kernel must record SIXBIT_EDEVICE, stop its other roles, wait for its own
copies and MMAs in flight, free its tensor memory and exit.  The host then
reads the error through sixbit_get_error(), and the next normal call on the
same stream must run and match the oracle.  No fault or hang is involved:
the wait that expires is the kernel's own bounded one."""
import time

import numpy as np
import pytest
import torch

import synthetic
from oracle import codecs, gemm as o_gemm, int8 as o_int8, nvfp4 as o_nvfp4
from tests.helpers import assert_gemm_close, dev, dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu


def _layer(residual):
    import nvfp4_int8_mixed_gb300 as sb
    M, K, N = 300, 256, 512                               # two 256-row CTA-pair tiles, a ragged M tail
    lay = synthetic.gemm_layer(21, M, K, N, residual)
    x = dev_bf16(lay["a"])
    wc, wsf, gw = sb.quantize_weight_nvfp4(dev(lay["w"]))
    codes, sf, ga = sb.quantize_act_nvfp4(x)
    _, planes, s = sb.quantize_act_int8(x, want_q=False)
    r = dev_bf16(lay["residual"]) if residual else None
    return lay, x, r, (wc, wsf, gw), (codes, sf, ga), (planes, s)


@pytest.mark.parametrize("residual", [False, True])
def test_expired_wait_reports_edevice_then_the_next_call_is_clean(residual):
    import nvfp4_int8_mixed_gb300 as sb
    lib = sb.lib()
    lay, x, r, (wc, wsf, gw), (codes, sf, ga), (planes, s) = _layer(residual)
    stream = sb._stream()
    assert lib.sixbit_get_error(stream) == sb.OK            # nothing pending before the test
    y = torch.empty((x.shape[0], wc.shape[0]), dtype=torch.bfloat16, device="cuda")
    assert lib.sixbit_debug_stall_gemm(1) == sb.OK
    try:
        for run in (lambda: sb.qlinear_w4a4(codes, sf, ga, wc, wsf, gw, residual=r, out=y),
                    lambda: sb.qlinear_w4a8(planes, s, wc, wsf, gw, residual=r, out=y)):
            t0 = time.perf_counter()
            run()                                          # the launch itself succeeds
            rc = lib.sixbit_get_error(stream)
            dt = time.perf_counter() - t0
            assert rc == sb.EDEVICE, rc
            assert dt < 60.0, dt                           # the wait gave up in bounded time
            print(f"expired wait reported after {dt:.2f} s")
            assert lib.sixbit_get_error(stream) == sb.OK   # reading the error cleared it
    finally:
        assert lib.sixbit_debug_stall_gemm(0) == sb.OK
    # the same stream runs normal layers again, with correct results
    af = codecs.bf16_to_f32(lay["a"])
    rwc, rwsf, rgw, _ = o_nvfp4.quantize(lay["w"])
    rac, rasf, rga, _ = o_nvfp4.quantize(af)
    rq, rs, _ = o_int8.quantize(af)
    y4 = sb.qlinear_w4a4(codes, sf, ga, wc, wsf, gw, residual=r, out_dtype=torch.float32)
    y8 = sb.qlinear_w4a8(planes, s, wc, wsf, gw, residual=r, out_dtype=torch.float32)
    assert lib.sixbit_get_error(stream) == sb.OK
    res = lay["residual"] if residual else None
    assert_gemm_close(host(y4), o_gemm.w4a4(rac, rasf, rga, rwc, rwsf, rgw, residual=res), "f32")
    assert_gemm_close(host(y8), o_gemm.w4a8(rq, rs, rwc, rwsf, rgw, residual=res), "f32")


@pytest.mark.parametrize("quant", [False, True])
def test_layernorm_expired_row_wait_reports_edevice_then_the_next_call_is_clean(quant):
    """The LayerNorm producer's row-prefetch form (bulk copies into shared
    memory, one bounded mbarrier wait a row): sixbit_debug_stall_staging(1)
    makes each warp wait for its first row on a barrier nothing signals.  The
    wait gives up, the kernel records SIXBIT_EDEVICE after letting its own
    row copies land, and the next normal call on the same stream is clean."""
    import nvfp4_int8_mixed_gb300 as sb
    from oracle import block as o_block
    lib = sb.lib()
    stream = sb._stream()
    # bf16 output with rows of 1920 (8-warp CTAs), or INT8 with rows of 3072 (4-warp CTAs):
    # both take the prefetch form
    M, H = (600, 3072) if quant else (600, 1920)
    x = synthetic.activations(synthetic.rng(M + H), M, H, 4, 10.0, 50.0)
    xd = dev_bf16(x)
    y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    planes = torch.empty((3, M, H // 2), dtype=torch.uint8, device="cuda")
    rs = torch.empty(M, device="cuda")
    run = (lambda: sb.layernorm_quant(xd, int8=(planes, rs))) if quant else (lambda: sb.layernorm(xd, out=y))
    assert lib.sixbit_get_error(stream) == sb.OK
    assert lib.sixbit_debug_stall_staging(1) == sb.OK
    try:
        t0 = time.perf_counter()
        run()                                              # the launch itself succeeds
        rc = lib.sixbit_get_error(stream)
        dt = time.perf_counter() - t0
        assert rc == sb.EDEVICE, rc
        assert dt < 60.0, dt                               # the waits gave up in bounded time
        print(f"expired row wait reported after {dt:.2f} s")
        assert lib.sixbit_get_error(stream) == sb.OK
    finally:
        assert lib.sixbit_debug_stall_staging(0) == sb.OK
    run()
    assert lib.sixbit_get_error(stream) == sb.OK
    ref = codecs.bf16_to_f32(o_block.layernorm(x)).astype(np.float64)
    if quant:
        got = host(rs).astype(np.float64)                  # row scales = |y| row max / 127
        want = np.max(np.abs(ref), axis=1) / 127.0
        assert np.all(np.abs(got - want) <= 2.0 ** -7 * want + 1e-9)
    else:
        got = codecs.bf16_to_f32(host_bf16_bits(y)).astype(np.float64)
        assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-6)


@pytest.mark.parametrize("mx", [False, True])
def test_gamma_expired_stage_wait_reports_edevice_then_the_next_call_is_clean(mx):
    """The Gamma passes stage their tiles through shared memory by bulk copies,
    one bounded mbarrier wait a tile.  With sixbit_debug_stall_staging(1)
    every CTA waits for its first tile on a barrier nothing signals: the wait
    gives up, the kernel records SIXBIT_EDEVICE after its own copies land and
    still completes its CTA count, so the next call on the same scratch and
    stream is clean and bit-exact."""
    import nvfp4_int8_mixed_gb300 as sb
    from oracle import gamma as o_gamma, mxcache
    lib = sb.lib()
    stream = sb._stream()
    M, H = 300, 1920                                       # 71 tiles of 8192 elements, the last one partial
    p = synthetic.gamma_pair(77, M, H)
    xin, xout = dev_bf16(p["xin"]), dev_bf16(p["xout"])
    ws = sb.workspace(int(lib.sixbit_workspace_size(M * H, 1)))
    if mx:
        codes, sc = mxcache.encode(codecs.bf16_to_f32(p["delta_prev"]))
        prev_bytes, prev_val = mxcache.to_bytes(codes, sc), mxcache.decode(codes, sc)
        fresh = lambda: dev(prev_bytes.copy())
    else:
        fresh = lambda: dev_bf16(p["delta_prev"])
    state = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    assert lib.sixbit_get_error(stream) == sb.OK
    assert lib.sixbit_debug_stall_staging(1) == sb.OK
    try:
        t0 = time.perf_counter()
        sb.block_gamma(xin, xout, delta=fresh(), tdc_state=state.clone(), ws=ws)
        rc = lib.sixbit_get_error(stream)
        dt = time.perf_counter() - t0
        assert rc == sb.EDEVICE, rc
        assert dt < 60.0, dt
        print(f"expired stage wait reported after {dt:.2f} s")
        assert lib.sixbit_get_error(stream) == sb.OK
    finally:
        assert lib.sixbit_debug_stall_staging(0) == sb.OK
    d = fresh()
    g, r2 = sb.block_gamma(xin, xout, delta=d, tdc_state=state, ws=ws)
    assert lib.sixbit_get_error(stream) == sb.OK
    rdn = o_gamma.delta(p["xin"], p["xout"])
    assert host(g)[0] == o_gamma.gamma(p["xin"], p["xout"])
    if mx:
        assert host(r2)[0] == o_gamma.rel_l2_sq(rdn, prev_val)
    else:
        assert host(r2)[0] == o_gamma.rel_l2_sq(rdn, p["delta_prev"])
        assert np.array_equal(host_bf16_bits(d), rdn)
    assert host(state).tolist() == [2, 0]
