"""GPU parity of the Gamma/Delta pass (a7), DMPQ (a8), TDC (a9) and the
block harness LayerNorm.  Delta bits, Gamma and r2 (both reduced by the
fixed tree the oracle defines), flags and skip decisions are bit-exact."""
import numpy as np
import pytest
import torch

import synthetic
from oracle import block as o_block, codecs, dmpq as o_dmpq, gamma as o_gamma, tdc as o_tdc
from tests.helpers import dev, dev_bf16, host, host_bf16_bits

pytestmark = pytest.mark.gpu


def _sb():
    import nvfp4_int8_mixed_gb300 as sb
    return sb


@pytest.mark.parametrize("M,H", [(256, 256), (1, 8), (1, 5), (2, 3), (3, 5000), (7, 333), (3, 8191), (17, 1920),
                                 (synthetic.M_2B, 1920)])          # n < 8: no whole group, an empty tile stage
def test_gamma_delta_r2(M, H):
    sb = _sb()
    p = synthetic.gamma_pair(M * 7 + H, M, H)
    xin, xout, dprev = dev_bf16(p["xin"]), dev_bf16(p["xout"]), dev_bf16(p["delta_prev"])
    state = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    g, r2 = sb.block_gamma(xin, xout, delta=dprev, tdc_state=state)
    torch.cuda.synchronize()
    rg = o_gamma.gamma(p["xin"], p["xout"])
    rdn = o_gamma.delta(p["xin"], p["xout"])
    rr2 = o_gamma.rel_l2_sq(rdn, p["delta_prev"])
    assert host(g)[0] == rg and host(r2)[0] == rr2
    assert np.array_equal(host_bf16_bits(dprev), rdn)
    assert host(state).tolist() == [2, 0]


@pytest.mark.parametrize("M,H", [(7, 333), (synthetic.M_2B, 1920)])
def test_gamma_with_caller_scratch(M, H):
    """The pass with its own scratch (`ws`, zeroed, sixbit_workspace_size(n, 1)
    bytes) matches the oracle bit for bit, twice in a row on the same
    scratch (the last CTA leaves its counter at zero for the next call)."""
    sb = _sb()
    p = synthetic.gamma_pair(M + 3 * H, M, H)
    ws = torch.zeros(int(sb.lib().sixbit_workspace_size(M * H, 1)), dtype=torch.uint8, device="cuda")
    rg = o_gamma.gamma(p["xin"], p["xout"])
    rdn = o_gamma.delta(p["xin"], p["xout"])
    rr2 = o_gamma.rel_l2_sq(rdn, p["delta_prev"])
    for _ in range(2):
        xin, xout, dprev = dev_bf16(p["xin"]), dev_bf16(p["xout"]), dev_bf16(p["delta_prev"])
        state = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
        g, r2 = sb.block_gamma(xin, xout, delta=dprev, tdc_state=state, ws=ws)
        torch.cuda.synchronize()
        assert host(g)[0] == rg and host(r2)[0] == rr2
        assert np.array_equal(host_bf16_bits(dprev), rdn)


def test_gamma_deterministic_and_skipped_block():
    sb = _sb()
    p = synthetic.gamma_pair(3, 1000, 333)
    xin, xout = dev_bf16(p["xin"]), dev_bf16(p["xout"])
    d = dev_bf16(p["delta_prev"])
    g1, _ = sb.block_gamma(xin, xout)
    g2, _ = sb.block_gamma(xin, xout)
    assert host(g1)[0] == host(g2)[0]
    # skipped block: Gamma only, Delta and r2 untouched, consec + 1
    state = torch.tensor([3, 0], dtype=torch.int32, device="cuda")
    computed = torch.zeros(1, dtype=torch.uint8, device="cuda")
    r2 = torch.full((1,), 0.123, device="cuda")
    g3, _ = sb.block_gamma(xin, xout, delta=d, r2_out=r2, tdc_state=state, computed=computed)
    assert host(g3)[0] == host(g1)[0]
    assert np.array_equal(host_bf16_bits(d), p["delta_prev"])
    assert np.float32(host(r2)[0]) == np.float32(0.123)
    assert host(state).tolist() == [3, 1]


def test_gamma_closed_forms_on_device():
    sb = _sb()
    x = synthetic.activations(synthetic.rng(1), 64, 64, 0, 1.0)
    x2 = codecs.f32_to_bf16(2 * codecs.bf16_to_f32(x))
    g0, _ = sb.block_gamma(dev_bf16(x), dev_bf16(x))
    g1, _ = sb.block_gamma(dev_bf16(x), dev_bf16(x2))
    assert host(g0)[0] == 0.0 and host(g1)[0] == 1.0


def test_dmpq_bit_exact():
    sb = _sb()
    g = synthetic.rng(11)
    nb = 30
    G = g.uniform(0, 0.4, nb).astype(np.float32)
    alpha = g.uniform(0.5, 1.5, 4 * nb).astype(np.float32)
    beta = g.uniform(0, 0.01, 4 * nb).astype(np.float32)
    lb = np.repeat(np.arange(nb), 4).astype(np.int32)
    p = o_dmpq.predict(G, alpha, beta, lb)
    tau = np.float32(np.quantile(p, 0.6))
    for step in (0, 5):
        st = torch.tensor([step], dtype=torch.int32, device="cuda")
        gates = torch.empty((4 * nb, 2), dtype=torch.uint8, device="cuda")
        f = sb.dmpq_assign(dev(G), dev(alpha), dev(beta), dev(lb), float(tau), st, gates=gates)
        ref = o_dmpq.assign(G, alpha, beta, lb, tau, step)
        assert np.array_equal(host(f), ref)
        assert np.array_equal(host(gates)[:, 0], ref) and np.array_equal(host(gates)[:, 1], 1 - ref)
    # a layer whose prediction equals tau exactly goes to INT8
    st = torch.tensor([1], dtype=torch.int32, device="cuda")
    f = sb.dmpq_assign(dev(G), dev(alpha), dev(beta), dev(lb), float(p[7]), st)
    assert host(f)[7] == 0


@pytest.mark.parametrize("fresh,consec,r2,tau,max_skip,refresh,step", [
    (2, 0, 0.001, 0.05, 1, 0, 0), (1, 0, 0.0, 0.05, 1, 0, 0), (2, 1, 0.001, 0.05, 1, 0, 0),
    (2, 0, 0.0025, 0.05, 1, 0, 0), (5, 1, 0.001, 0.05, 2, 0, 0), (2, 0, 0.001, 0.0, 1, 0, 0),
    (2, 0, np.inf, 0.05, 1, 0, 0),
    # periodic refresh (PDR variant): step % k == 0 forces a computed step
    (2, 0, 0.001, 0.05, 1, 3, 6), (2, 0, 0.001, 0.05, 1, 3, 7), (5, 1, 0.001, 0.05, 2, 4, 9), (5, 1, 0.001, 0.05, 2, 4, 12)])
def test_tdc_decide_and_apply(fresh, consec, r2, tau, max_skip, refresh, step):
    sb = _sb()
    M, H = 37, 104
    p = synthetic.gamma_pair(4, M, H)
    xin, dl = dev_bf16(p["xin"]), dev_bf16(p["delta_prev"])
    state = torch.tensor([fresh, consec], dtype=torch.int32, device="cuda")
    cflag = torch.full((1,), 7, dtype=torch.uint8, device="cuda")
    out = torch.zeros((M, H), dtype=torch.bfloat16, device="cuda")
    gates = torch.ones(8, dtype=torch.uint8, device="cuda")
    step_t = torch.tensor([step], dtype=torch.int32, device="cuda")
    sb.tdc_decide_and_apply(xin, dl, torch.tensor([np.float32(r2)], device="cuda"), tau, max_skip, state, cflag, out,
                            gates=gates, refresh_every=refresh, step=step_t)
    cache = o_tdc.BlockCache(fresh_count=fresh, consec=consec, r2=np.float32(r2))
    skip = o_tdc.decide(cache, tau, max_skip, refresh, step)
    assert host(cflag)[0] == (0 if skip else 1)
    assert host(state).tolist() == [fresh, consec]           # counters advance in the Gamma pass
    if skip:
        assert np.array_equal(host_bf16_bits(out), o_tdc.apply(p["xin"], p["delta_prev"]))
        assert not host(gates).any()
    else:
        assert not host_bf16_bits(out).any() and host(gates).all()


@pytest.mark.parametrize("M,H", [(256, 256), (17776, 1920), (5, 3072), (17776, 1024), (6000, 4096)])
def test_layernorm(M, H):
    sb = _sb()
    x = synthetic.activations(synthetic.rng(M), M, H, 2, 30.0)
    amax = torch.empty(1, device="cuda")
    ramax = torch.empty(M, device="cuda")
    y = sb.layernorm(dev_bf16(x), amax_out=amax, row_amax_out=ramax)
    got = codecs.bf16_to_f32(host_bf16_bits(y)).astype(np.float64)
    rows = np.arange(M) if M <= 512 else np.random.default_rng(0).choice(M, 256, replace=False)
    ref = codecs.bf16_to_f32(o_block.layernorm(x[rows])).astype(np.float64)
    # float32 statistics vs float64: at most one bf16 ulp (2^-7 relative) apart
    assert np.all(np.abs(got[rows] - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-6)
    assert host(amax)[0] == np.max(np.abs(got))
    assert np.array_equal(host(ramax), np.max(np.abs(got), axis=1).astype(np.float32))


# ------------------------------------------- compressed update cache (MX)
def _mx_prev(p):
    from oracle import mxcache
    codes, sc = mxcache.encode(codecs.bf16_to_f32(p["delta_prev"]))
    return mxcache.to_bytes(codes, sc), mxcache.decode(codes, sc)


@pytest.mark.parametrize("M,H", [(256, 256), (1, 32), (3, 8192 + 96), (synthetic.M_2B, 1920)])
def test_gamma_mxcache_parity(M, H):
    from oracle import mxcache
    sb = _sb()
    p = synthetic.gamma_pair(M * 5 + H, M, H)
    prev_bytes, prev_val = _mx_prev(p)
    cache = dev(prev_bytes)
    assert cache.numel() == sb.lib().sixbit_mxcache_bytes(M * H)
    xin, xout = dev_bf16(p["xin"]), dev_bf16(p["xout"])
    state = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    g, r2 = sb.block_gamma(xin, xout, delta=cache, tdc_state=state)
    rdn = o_gamma.delta(p["xin"], p["xout"])
    rr2 = o_gamma.rel_l2_sq(rdn, prev_val.reshape(M, H))
    rg = o_gamma.gamma(p["xin"], p["xout"])
    assert host(g)[0] == rg and host(r2)[0] == rr2
    codes, sc = mxcache.encode(codecs.bf16_to_f32(rdn))
    assert np.array_equal(host(cache), mxcache.to_bytes(codes, sc))       # the new update, encoded
    assert host(state).tolist() == [2, 0]
    # a first update (no previous one): no r2, the cache is written
    c2 = torch.zeros_like(cache)
    r2b = torch.full((1,), 0.5, device="cuda")
    st0 = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    sb.block_gamma(xin, xout, delta=c2, r2_out=r2b, tdc_state=st0)
    assert np.array_equal(host(c2), host(cache)) and host(r2b)[0] == 0.5
    # a skipped block leaves the cache alone
    c3 = dev(prev_bytes)
    sb.block_gamma(xin, xout, delta=c3, tdc_state=state, computed=torch.zeros(1, dtype=torch.uint8, device="cuda"))
    assert np.array_equal(host(c3), prev_bytes)


@pytest.mark.parametrize("n", [32, 8192 * 3 + 64, synthetic.M_2B * 1920])
def test_tdc_mxcache_skip_output(n):
    from oracle import mxcache
    sb = _sb()
    g = synthetic.rng(n % 1000)
    xin = codecs.f32_to_bf16(g.standard_normal(n).astype(np.float32))
    d = codecs.f32_to_bf16((0.05 * g.standard_normal(n)).astype(np.float32))
    d[:32] = 0                                                            # a zero block
    codes, sc = mxcache.encode(codecs.bf16_to_f32(d))
    cache = dev(mxcache.to_bytes(codes, sc))
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    state = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    r2 = torch.tensor([1e-6], device="cuda")
    cflag = torch.empty(1, dtype=torch.uint8, device="cuda")
    gates = torch.ones(8, dtype=torch.uint8, device="cuda")
    sb.tdc_decide_and_apply(dev_bf16(xin), cache, r2, 0.05, 1, state, cflag, out, gates=gates)
    assert host(cflag)[0] == 0 and not host(gates).any()
    ref = o_tdc.apply(xin, mxcache.decode(codes, sc))
    assert np.array_equal(host_bf16_bits(out), ref)
