"""Pins of Gamma / Delta / r2, the DMPQ assignment and the TDC state machine."""
import numpy as np

from oracle import codecs, dmpq, gamma, tdc
from oracle.codecs import f32_to_bf16


def _bits(x):
    return f32_to_bf16(np.asarray(x, np.float32))


def test_gamma_closed_forms():
    rng = np.random.default_rng(0)
    x = _bits(rng.standard_normal((7, 33)))
    assert gamma.gamma(x, x) == 0.0
    x2 = _bits(2 * codecs.bf16_to_f32(x))
    assert gamma.gamma(x, x2) == 1.0                      # power-of-two scaling is exact
    c = _bits(np.full((4, 10), 0.5))
    c3 = _bits(np.full((4, 10), 2.0))
    assert gamma.gamma(c, c3) == np.float32(3.0)           # |2 - 0.5| / 0.5
    z = _bits(np.zeros((3, 3)))
    assert gamma.gamma(z, c[:3, :3]) == 0.0                # ||in|| = 0 -> 0 by definition


def _scalar_tree(terms):
    """The reduction tree of oracle.gamma walked one element at a time (float32
    lanes, float64 across tiles), written independently of the vectorised
    version it checks."""
    terms = [np.float32(v) for v in terms]
    n = len(terms)
    tile_sums = []
    for base in range(0, max(n, 1), 8192):
        lanes = []
        for t in range(256):
            acc = np.float32(0.0)
            for j in range(4):
                for e in range(8):
                    i = base + j * 2048 + 8 * t + e
                    if i < n:
                        acc = np.float32(acc + terms[i])
            lanes.append(acc)
        for h in (16, 8, 4, 2, 1):
            lanes = [np.float32(lanes[k] + lanes[k ^ h]) for k in range(256)]
        groups = [lanes[32 * w] for w in range(8)]
        for h in (4, 2, 1):
            for w in range(h):
                groups[w] = np.float32(groups[w] + groups[w + h])
        tile_sums.append(float(groups[0]))
    acc = [0.0] * 256
    for k, v in enumerate(tile_sums):
        acc[k % 256] = acc[k % 256] + v
    h = 128
    while h >= 1:
        for k in range(h):
            acc[k] = acc[k] + acc[k + h]
        h //= 2
    return acc[0]


def test_tree_sum_matches_a_scalar_walk_of_the_tree():
    rng = np.random.default_rng(7)
    # magnitudes over 12 binades, so the float32 result depends on the order
    n = 2 * 8192 + 1003
    v = (rng.standard_normal(n) ** 2 * np.exp2(rng.integers(-6, 6, n))).astype(np.float32)
    got = gamma.tree_sum(v)
    assert got == _scalar_tree(v)
    # a different order (one float32 running sum, or float64 throughout) gives other bits
    seq = np.float32(0.0)
    for x in v:
        seq = np.float32(seq + x)
    assert float(seq) != got and float(np.sum(v.astype(np.float64))) != got
    assert gamma.tree_sum(v[:5]) == _scalar_tree(v[:5])


def test_tree_sum_closed_forms_and_bound():
    assert gamma.tree_sum(np.ones(8192, np.float32)) == 8192.0
    assert gamma.tree_sum(np.ones(3 * 8192 + 5, np.float32)) == 3 * 8192 + 5
    assert gamma.tree_sum(np.zeros(10, np.float32)) == 0.0
    # 300 tiles: more tiles than float64 lanes, so lanes add several tiles
    assert gamma.tree_sum(np.full(300 * 8192, 0.5, np.float32)) == 300 * 4096
    rng = np.random.default_rng(8)
    v = np.abs(rng.standard_normal(1_000_003)).astype(np.float32)
    exact = float(np.sum(v.astype(np.float64)))
    # nonnegative terms: 31 sequential float32 adds per lane, 8 tree levels
    assert abs(gamma.tree_sum(v) - exact) <= 40 * 2.0 ** -24 * exact


def test_gamma_and_r2_within_rounding_of_the_exact_values():
    rng = np.random.default_rng(9)
    xin = _bits(rng.standard_normal((37, 1000)))
    xout = _bits(codecs.bf16_to_f32(xin) + 0.05 * rng.standard_normal((37, 1000)))
    g, ge = gamma.gamma(xin, xout), gamma.gamma_exact(xin, xout)
    assert g != 0 and abs(g - ge) <= 1e-5 * ge
    dn = gamma.delta(xin, xout)
    dp = _bits(codecs.bf16_to_f32(dn) * (1 + 0.1 * rng.standard_normal((37, 1000))))
    r, re = gamma.rel_l2_sq(dn, dp), gamma.rel_l2_sq_exact(dn, dp)
    assert r != 0 and abs(r - re) <= 1e-5 * re


def test_delta_and_r2_closed_forms():
    rng = np.random.default_rng(1)
    xin = _bits(rng.standard_normal((5, 16)))
    d = _bits(rng.standard_normal((5, 16)) * 0.1)
    xout = _bits(codecs.bf16_to_f32(xin) + codecs.bf16_to_f32(d))
    dn = gamma.delta(xin, xout)
    assert gamma.rel_l2_sq(dn, dn) == 0.0
    d2 = _bits(2 * codecs.bf16_to_f32(dn))
    assert gamma.rel_l2_sq(d2, dn) == 1.0                  # ||2D - D|| / ||D|| = 1
    assert gamma.rel_l2_sq(dn, _bits(np.zeros((5, 16)))) == np.inf
    assert abs(gamma.cosine(d2, dn) - 1.0) < 1e-12
    assert abs(gamma.cosine(_bits(-codecs.bf16_to_f32(dn)), dn) + 1.0) < 1e-12


def test_delta_is_f32_difference_rounded_to_bf16():
    xin = _bits([[1.0, 3.0, -2.0]])
    xout = _bits([[1.5, 3.015625, 2.0]])
    assert codecs.bf16_to_f32(gamma.delta(xin, xout)).tolist() == [[0.5, 0.015625, 4.0]]


def test_block_pass_contract():
    rng = np.random.default_rng(2)
    xin = _bits(rng.standard_normal((3, 8)))
    xout = _bits(rng.standard_normal((3, 8)))
    g, dn, r2 = gamma.block_pass(xin, xout, None, computed=True)
    assert dn is not None and r2 is None
    g2, dn2, r22 = gamma.block_pass(xin, xout, dn, computed=True)
    assert g2 == g and r22 == 0.0
    g3, dn3, r23 = gamma.block_pass(xin, xout, dn, computed=False)
    assert g3 == g and dn3 is None and r23 is None


def test_dmpq_extremes_reproduce_uniform_policies():
    rng = np.random.default_rng(3)
    G = rng.uniform(0, 0.5, 6).astype(np.float32)
    alpha = rng.uniform(0.5, 1.5, 24).astype(np.float32)
    beta = rng.uniform(0, 0.01, 24).astype(np.float32)
    lb = np.repeat(np.arange(6), 4)
    assert dmpq.assign(G, alpha, beta, lb, np.inf, 3).all()             # uniform W4A4
    assert not dmpq.assign(G, alpha, beta, lb, -np.inf, 3).any()        # uniform W4A8
    assert not dmpq.assign(G, alpha, beta, lb, np.inf, 0).any()         # step 0 -> INT8
    f = dmpq.assign(G, np.zeros(24, np.float32), beta, lb, np.float32(0.005), 2)
    assert np.array_equal(f, (beta < np.float32(0.005)).astype(np.uint8))


def test_dmpq_tie_goes_to_int8_and_layer_block_map():
    G = np.array([0.25, 0.5], np.float32)
    alpha = np.array([1.0, 1.0, 2.0], np.float32)
    beta = np.array([0.0, 0.25, 0.0], np.float32)
    lb = np.array([0, 0, 1])
    p = dmpq.predict(G, alpha, beta, lb)
    assert p.tolist() == [0.25, 0.5, 1.0]
    assert dmpq.assign(G, alpha, beta, lb, 0.5, 1).tolist() == [1, 0, 0]


def test_dmpq_calibration_fraction():
    p = np.arange(1000, dtype=np.float32)
    tau = dmpq.calibrate_tau(p, 0.6)
    assert abs(np.mean(p < tau) - 0.6) < 0.002


def test_tdc_state_machine_hand_sequence():
    # r2 values as produced by consecutive computed steps; tau 0.05 -> tau^2 = 0.0025
    c = tdc.BlockCache()
    seq = []
    r2_next = [None, 0.001, 0.001, 0.01, 0.0001, 0.0001]
    i = 0
    for step in range(8):
        if tdc.decide(c, 0.05, 1):
            tdc.after_skip(c)
            seq.append("S")
        else:
            tdc.after_compute(c, np.zeros(1, np.uint16), r2_next[i])
            i += 1
            seq.append("C")
    # C (first delta) C (r2 .001, 2 fresh) S C (r2 .001, consec reset) S C (r2 .01) C (r2 1e-4) S
    assert "".join(seq) == "CCSCSCCS"


def test_tdc_pdr_variants_hand_sequences():
    # every computed step yields r2 = 1e-4 < tau^2: skips are limited only by
    # fresh_count, max_skip and the periodic refresh
    def run(max_skip, refresh_every, steps=12):
        c = tdc.BlockCache()
        seq = []
        for t in range(steps):
            if tdc.decide(c, 0.05, max_skip, refresh_every, t):
                tdc.after_skip(c)
                seq.append("S")
            else:
                tdc.after_compute(c, np.zeros(1, np.uint16), 1e-4 if c.delta is not None else None)
                seq.append("C")
        return "".join(seq)
    assert run(1, 0) == "CCSCSCSCSCSC"          # max_skip 1 alternates after two fresh updates
    assert run(2, 0) == "CCSSCSSCSSCS"          # two reuses between computed steps
    # refresh every 4 steps: t = 0, 4, 8 computed whatever the rule says
    assert run(2, 4) == "CCSSCSSCCSSC"
    assert run(1, 3) == "CCSCSCCSCCSC"


def test_tdc_never_skips_with_zero_threshold_or_zero_max_skip():
    c = tdc.BlockCache(fresh_count=5, consec=0, r2=np.float32(0.0), delta=None)
    assert not tdc.decide(c, 0.0, 1)                      # r2 < 0 is impossible
    assert not tdc.decide(c, 1.0, 0)
    assert tdc.decide(c, 1.0, 1)


def test_tdc_needs_two_computed_updates():
    # r2 compares the updates of two computed steps, so a block with only one
    # computed update is never skipped, even when the caller's r2 is below
    # the threshold (a state the device contract accepts as input)
    one = tdc.BlockCache(fresh_count=1, consec=0, r2=np.float32(0.0), delta=None)
    two = tdc.BlockCache(fresh_count=2, consec=0, r2=np.float32(0.0), delta=None)
    assert not tdc.decide(one, 0.05, 1)
    assert tdc.decide(two, 0.05, 1)


def test_tdc_apply_identity():
    rng = np.random.default_rng(4)
    xin = _bits(rng.standard_normal((6, 40)))
    d = _bits(rng.standard_normal((6, 40)) * 0.05)
    out = tdc.apply(xin, d)
    back = codecs.bf16_to_f32(out).astype(np.float64) - codecs.bf16_to_f32(xin)
    ulp = np.abs(codecs.bf16_to_f32(out)).astype(np.float64) * 2.0 ** -8
    assert (np.abs(back - codecs.bf16_to_f32(d)) <= ulp + 1e-30).all()
    assert np.array_equal(tdc.apply(xin, _bits(np.zeros((6, 40)))), xin)
