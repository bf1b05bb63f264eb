"""Planted mistakes in the oracle, each of which the oracle's pins must catch.

Every case below replaces one oracle function (or one constant or library
call inside it) with a version that carries a single plausible error: a
dropped term, a wrong rounding rule, a swapped operand or index, an
off-by-one in a decision.  It then runs the pin tests that cover that part
of the oracle and requires at least one of them to fail.  A mistake that no
pin detects is a gap in the pins, so this file guards the claim that the
oracle is checked against something other than itself.  CPU only; the
oracle modules are patched through pytest's monkeypatch and restored after
each case.
"""
import importlib
import sys

import numpy as np
import pytest

from oracle import block, calib, codecs, dmpq, gamma, gemm, int8, mxcache, nvfp4, tdc

F32 = np.float32


def _pins(*names):
    """'module.function' names of pin tests in tests/test_oracle_<module>.py."""
    out = []
    for n in names:
        mod, fn = n.split(".")
        out.append((n, getattr(importlib.import_module("tests.test_oracle_" + mod), fn)))
    return out


def _replace(mp, old, new):
    """Point every reference to `old` in the loaded oracle and test modules at
    `new` (modules import each other's functions by name)."""
    for name, m in list(sys.modules.items()):
        if m is None or not (name == "oracle" or name.startswith(("oracle.", "tests.", "test_oracle"))):
            continue
        for attr, val in list(vars(m).items()):
            if val is old:
                mp.setattr(m, attr, new)


class _Np:
    """numpy with a few functions overridden, for patching `np` in one module."""

    def __init__(self, **over):
        self.__dict__.update(over)

    def __getattr__(self, name):
        return getattr(np, name)


# ------------------------------------------------------------------ codecs
_E2M1_MID = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])   # midpoints of the E2M1 magnitudes


def e2m1_ties_down(mp):
    real = codecs.e2m1_encode

    def enc(v):
        c = real(v)
        a = np.abs(np.asarray(v, dtype=F32)).astype(np.float64)
        mid = np.isin(a, _E2M1_MID)
        lower = np.searchsorted(_E2M1_MID, a).astype(np.uint8)   # the smaller neighbour's code
        return np.where(mid, (c & 8) | lower, c).astype(np.uint8)
    _replace(mp, real, enc)


def pack_high_nibble_first(mp):
    def pack(codes):
        c = np.asarray(codes, dtype=np.uint8)
        return ((c[..., 0::2] & 0xF) << 4) | (c[..., 1::2] & 0xF)
    _replace(mp, codecs.pack_e2m1, pack)


def e4m3_truncates(mp):
    mags = codecs.e4m3_decode(np.arange(0x7F)).astype(np.float64)

    def enc(v):
        v = np.asarray(v, dtype=F32)
        flat = v.reshape(-1)
        idx = np.clip(np.searchsorted(mags, np.abs(flat.astype(np.float64)), side="right") - 1, 0, len(mags) - 1)
        return (idx + np.where(np.signbit(flat), 0x80, 0)).astype(np.uint8).reshape(v.shape)
    _replace(mp, codecs.e4m3_encode, enc)


def e4m3_overflows_to_nan(mp):
    real = codecs.e4m3_encode

    def enc(v):
        c = real(v)
        big = np.abs(np.asarray(v, dtype=F32)) >= 464.0          # past the last rounding interval of 448
        return np.where(big, c | 0x7F, c).astype(np.uint8)
    _replace(mp, real, enc)


def bf16_truncates(mp):
    def to_bf16(x):
        x = np.ascontiguousarray(np.asarray(x, dtype=F32))
        return (x.view(np.uint32) >> 16).astype(np.uint16)
    _replace(mp, codecs.f32_to_bf16, to_bf16)


# ------------------------------------------------------------------ NVFP4
def global_scale_without_e2m1_max(mp):
    def gs(amax_t):
        a = F32(amax_t)
        return F32(1.0) if a == 0 else F32(a / F32(448.0))
    _replace(mp, nvfp4.global_scale, gs)


def block_scale_without_448(mp):
    mp.setattr(nvfp4, "E4M3_MAX", 1.0)                           # s_b = amax_b / amax_t, g = amax_t / 6


def sf_layout_row_major_atom(mp):
    def off(m, c, kc4):
        m = np.asarray(m, dtype=np.int64)
        c = np.asarray(c, dtype=np.int64)
        return ((m // 128) * (kc4 // 4) + c // 4) * 512 + (m % 128) * 4 + c % 4
    _replace(mp, nvfp4.sf_offset, off)


def delayed_ignores_headroom(mp):
    real = nvfp4.quantize

    def qd(x, amax_prev, headroom=2.0):
        codes, sf, g, _ = real(x, F32(amax_prev))
        return codes, sf, g, F32(amax_prev), nvfp4.tensor_amax(x)
    _replace(mp, nvfp4.quantize_delayed, qd)


# ------------------------------------------------------------------ INT8
def int8_round_half_away(mp):
    mp.setattr(int8, "np", _Np(rint=lambda v: np.sign(v) * np.floor(np.abs(v) + 0.5)))


def int8_clamps_at_minus_128(mp):
    mp.setattr(int8, "np", _Np(clip=lambda v, lo, hi: np.clip(v, -128 if lo == -127 else lo, hi)))


def digits_not_centred(mp):
    def digits(q):
        q = np.asarray(q, dtype=np.int64)
        c = q % 8
        q1 = (q - c) // 8
        b = q1 % 8
        return (q1 - b) // 8, b, c
    _replace(mp, int8.digits, digits)


# ------------------------------------------------------------------ GEMM
def w4a4_drops_activation_scale(mp):
    real = gemm.w4a4

    def w(a_codes, a_sf, g_a, *args, **kw):
        return real(a_codes, a_sf, 1.0, *args, **kw)
    _replace(mp, real, w)


def w4a8_row_scales_reversed(mp):
    real = gemm.w4a8

    def w(q, s_a, *args, **kw):
        return real(q, np.asarray(s_a)[::-1], *args, **kw)
    _replace(mp, real, w)


def epilogue_residual_before_gelu(mp):
    def epi(acc, bias=None, gelu=False, residual=None, out_dtype="f32"):
        y = np.asarray(acc, dtype=np.float64)
        if bias is not None:
            y = y + codecs.bf16_to_f32(bias).astype(np.float64)[None, :]
        if residual is not None:
            y = y + codecs.bf16_to_f32(residual).astype(np.float64)
        if gelu:
            y = gemm.gelu_tanh(y)
        return y.astype(np.float32) if out_dtype == "f32" else codecs.f64_to_bf16(y)
    _replace(mp, gemm.epilogue, epi)


def gelu_wrong_constant(mp):
    mp.setattr(gemm, "SQRT_2_OVER_PI", np.sqrt(2.0) / np.pi)


def layernorm_without_centring(mp):
    def ln(x_bits, eps=block.LN_EPS):
        x = codecs.bf16_to_f32(x_bits).astype(np.float64)
        mu = x.mean(axis=1, keepdims=True)
        var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
        return codecs.f64_to_bf16(x / np.sqrt(var + eps))
    _replace(mp, block.layernorm, ln)


# ------------------------------------------------------------------ Gamma / r2
def gamma_over_output_norm(mp):
    def g(xin, xout):
        fi = codecs.bf16_to_f32(xin).astype(F32).ravel()
        fo = codecs.bf16_to_f32(xout).astype(F32).ravel()
        d = (fo - fi).astype(F32)
        return gamma._ratio(gamma.tree_sum(np.abs(d)), gamma.tree_sum(np.abs(fo)), F32(0.0))
    _replace(mp, gamma.gamma, g)


def tree_sum_drops_ragged_tail(mp):
    real = gamma.tree_sum

    def ts(terms):
        t = np.asarray(terms, dtype=F32).ravel()
        n = (t.size // gamma.TILE) * gamma.TILE
        return real(t[:n]) if n else real(t)
    _replace(mp, real, ts)


def _tree_sum_variant(warp_serial=False, contiguous_lanes=False):
    """The oracle's reduction tree with one step reordered."""
    T, L, V = gamma.TILE, gamma.LANES, gamma.VEC

    def ts(terms):
        t = np.asarray(terms, dtype=F32).ravel()
        ntiles = max(1, -(-t.size // T))
        p = np.zeros(ntiles * T, dtype=F32)
        p[:t.size] = t
        if contiguous_lanes:                   # lane k adds elements 32k .. 32k + 31 of the tile
            x = p.reshape(ntiles, L, T // L).transpose(0, 2, 1)
        else:                                  # lane k adds elements j*2048 + 8k + e
            x = p.reshape(ntiles, T // (L * V), L, V).transpose(0, 1, 3, 2).reshape(ntiles, T // L, L)
        lane = np.zeros((ntiles, L), dtype=F32)
        for i in range(x.shape[1]):
            lane = (lane + x[:, i, :]).astype(F32)
        g = lane.reshape(ntiles, L // 32, 32)
        if warp_serial:                        # the 32 lanes added one after another
            acc32 = g[:, :, 0].copy()
            for k in range(1, 32):
                acc32 = (acc32 + g[:, :, k]).astype(F32)
            g[:, :, 0] = acc32
        else:
            idx = np.arange(32)
            for h in (16, 8, 4, 2, 1):
                g = (g + g[:, :, idx ^ h]).astype(F32)
        w = g[:, :, 0].copy()
        for h in (4, 2, 1):
            w[:, :h] = (w[:, :h] + w[:, h:2 * h]).astype(F32)
        tiles = w[:, 0].astype(np.float64)
        nb = -(-ntiles // L)
        tp = np.zeros(nb * L)
        tp[:ntiles] = tiles
        acc = np.zeros(L)
        for b in range(nb):                    # lane k adds tiles k, k + 256, ... in order
            acc = acc + tp[b * L:(b + 1) * L]
        h = L // 2
        while h >= 1:
            acc[:h] = acc[:h] + acc[h:2 * h]
            h //= 2
        return np.float64(acc[0])
    return ts


def tree_warp_serial(mp):
    _replace(mp, gamma.tree_sum, _tree_sum_variant(warp_serial=True))


def tree_contiguous_lanes(mp):
    _replace(mp, gamma.tree_sum, _tree_sum_variant(contiguous_lanes=True))


def r2_denominator_not_squared(mp):
    def r2(delta_new, delta_prev):
        dn, dp = gamma._f32(delta_new), gamma._f32(delta_prev)
        e = (dn - dp).astype(F32)
        return gamma._ratio(gamma.tree_sum((e * e).astype(F32)), gamma.tree_sum(np.abs(dp)), F32(np.inf))
    _replace(mp, gamma.rel_l2_sq, r2)


# ------------------------------------------------------------------ DMPQ / TDC
def dmpq_tie_goes_to_nvfp4(mp):
    def assign(gamma_blocks, alpha, beta, layer_block, tau, step):
        if step == 0:
            return np.zeros(len(alpha), dtype=np.uint8)
        return (dmpq.predict(gamma_blocks, alpha, beta, layer_block) <= F32(tau)).astype(np.uint8)
    _replace(mp, dmpq.assign, assign)


def dmpq_step0_not_forced(mp):
    def assign(gamma_blocks, alpha, beta, layer_block, tau, step):
        return (dmpq.predict(gamma_blocks, alpha, beta, layer_block) < F32(tau)).astype(np.uint8)
    _replace(mp, dmpq.assign, assign)


def tdc_max_skip_off_by_one(mp):
    def decide(cache, tau_tdc, max_skip, refresh_every=0, step=0):
        if refresh_every > 0 and step % refresh_every == 0:
            return False
        t2 = F32(F32(tau_tdc) * F32(tau_tdc))
        return cache.fresh_count >= 2 and F32(cache.r2) < t2 and cache.consec <= max_skip
    _replace(mp, tdc.decide, decide)


def tdc_threshold_not_squared(mp):
    def decide(cache, tau_tdc, max_skip, refresh_every=0, step=0):
        if refresh_every > 0 and step % refresh_every == 0:
            return False
        return cache.fresh_count >= 2 and F32(cache.r2) < F32(tau_tdc) and cache.consec < max_skip
    _replace(mp, tdc.decide, decide)


def tdc_one_fresh_step_suffices(mp):
    def decide(cache, tau_tdc, max_skip, refresh_every=0, step=0):
        if refresh_every > 0 and step % refresh_every == 0:
            return False
        t2 = F32(F32(tau_tdc) * F32(tau_tdc))
        return cache.fresh_count >= 1 and F32(cache.r2) < t2 and cache.consec < max_skip
    _replace(mp, tdc.decide, decide)


def tdc_apply_subtracts(mp):
    def apply(xin, delta_fresh):
        d = np.asarray(delta_fresh)
        df = codecs.bf16_to_f32(d) if d.dtype == np.uint16 else d.astype(F32)
        return codecs.f32_to_bf16((codecs.bf16_to_f32(xin) - df).astype(F32))
    _replace(mp, tdc.apply, apply)


# ------------------------------------------------------------------ block and stack
def qlinear_ignores_flag_int8(mp):
    real = block.qlinear

    def ql(h_bits, wq, use_nvfp4, **kw):
        return real(h_bits, wq, False, **kw)
    _replace(mp, real, ql)


def qlinear_ignores_flag_nvfp4(mp):
    real = block.qlinear

    def ql(h_bits, wq, use_nvfp4, **kw):
        return real(h_bits, wq, True, **kw)
    _replace(mp, real, ql)


def dmpq_never_picks_nvfp4(mp):
    def assign(gamma_blocks, alpha, beta, layer_block, tau, step):
        return np.zeros(len(alpha), dtype=np.uint8)
    _replace(mp, dmpq.assign, assign)


# ------------------------------------------------------------------ compressed cache / calibration
def mx_scale_exponent_one_low(mp):
    real = mxcache.scale_exponent

    def k(amax):
        a = np.asarray(amax, dtype=np.float64)
        return np.where(a == 0, real(a), real(a) - 1)
    _replace(mp, real, k)


def mx_layout_scales_first(mp):
    def to_bytes(codes, scales):
        return np.concatenate([np.asarray(scales, np.uint8).reshape(-1), np.asarray(codes, np.uint8).reshape(-1)])
    _replace(mp, mxcache.to_bytes, to_bytes)


def r_squared_complement(mp):
    real = calib.r_squared

    def r2(x, y, alpha, beta):
        return 1.0 - real(x, y, alpha, beta)
    _replace(mp, real, r2)


def fit_line_swapped(mp):
    real = calib.fit_line

    def fit(x, y):
        a, b = real(x, y)
        return b, a
    _replace(mp, real, fit)


def cosine_without_sqrt(mp):
    def cos(a, b):
        s = calib.pair_sums(a, b)
        den = s[3] * s[1]
        return 0.0 if den == 0.0 else float(s[2] / den)
    _replace(mp, calib.cosine, cos)


MUTANTS = [
    (e2m1_ties_down, ("codecs.test_e2m1_rounding_fixture", "codecs.test_e2m1_nearest_brute_force")),
    (pack_high_nibble_first, ("codecs.test_e2m1_pack_low_nibble_first",)),
    (bf16_truncates, ("codecs.test_bf16_vs_torch", "gemm.test_bf16_output_is_rounded_f32")),
    (e4m3_truncates, ("codecs.test_e4m3_encode_vs_torch_in_range", "codecs.test_e4m3_fixture_points")),
    (e4m3_overflows_to_nan, ("quant.test_caller_amax_below_true_amax_saturates",)),
    (global_scale_without_e2m1_max, ("quant.test_block_at_tensor_amax_gets_max_scale",
                                     "quant.test_known_scales_recover_grid_exactly")),
    (block_scale_without_448, ("quant.test_block_at_tensor_amax_gets_max_scale",
                               "quant.test_known_scales_recover_grid_exactly")),
    (sf_layout_row_major_atom, ("quant.test_sf_layout_fixed_points_and_bijection",)),
    (delayed_ignores_headroom, ("delayed.test_grown_amax_saturates_at_the_used_amax",
                                "delayed.test_power_of_two_headroom_keeps_the_dequantized_tensor")),
    (int8_round_half_away, ("quant.test_int8_ties_to_even",)),
    (int8_clamps_at_minus_128, ("quant.test_int8_saturates_with_small_caller_amax",
                                "quant.test_int8_extremes_and_zero_row")),
    (digits_not_centred, ("quant.test_digit_split_reconstructs_every_code",)),
    (w4a4_drops_activation_scale, ("gemm.test_w4a4_matches_triple_loop",)),
    (w4a8_row_scales_reversed, ("gemm.test_w4a8_matches_triple_loop",)),
    (epilogue_residual_before_gelu, ("gemm.test_w4a4_matches_triple_loop", "gemm.test_w4a8_matches_triple_loop",
                                     "block.test_block_residual_wiring_with_zero_weights")),
    (gelu_wrong_constant, ("gemm.test_gelu_vs_torch",)),
    (layernorm_without_centring, ("block.test_layernorm_vs_torch",)),
    (gamma_over_output_norm, ("gamma_dmpq_tdc.test_gamma_closed_forms",)),
    (tree_sum_drops_ragged_tail, ("gamma_dmpq_tdc.test_tree_sum_matches_a_scalar_walk_of_the_tree",
                                  "gamma_dmpq_tdc.test_tree_sum_closed_forms_and_bound")),
    (tree_warp_serial, ("gamma_dmpq_tdc.test_tree_sum_matches_a_scalar_walk_of_the_tree",)),
    (tree_contiguous_lanes, ("gamma_dmpq_tdc.test_tree_sum_matches_a_scalar_walk_of_the_tree",)),
    (r2_denominator_not_squared, ("gamma_dmpq_tdc.test_delta_and_r2_closed_forms",)),
    (dmpq_tie_goes_to_nvfp4, ("gamma_dmpq_tdc.test_dmpq_tie_goes_to_int8_and_layer_block_map",)),
    (dmpq_step0_not_forced, ("gamma_dmpq_tdc.test_dmpq_extremes_reproduce_uniform_policies",
                             "gamma_dmpq_tdc.test_dmpq_tie_goes_to_int8_and_layer_block_map")),
    (tdc_max_skip_off_by_one, ("gamma_dmpq_tdc.test_tdc_state_machine_hand_sequence",
                               "gamma_dmpq_tdc.test_tdc_never_skips_with_zero_threshold_or_zero_max_skip")),
    (tdc_threshold_not_squared, ("gamma_dmpq_tdc.test_tdc_state_machine_hand_sequence",
                                 "gamma_dmpq_tdc.test_tdc_pdr_variants_hand_sequences")),
    (tdc_one_fresh_step_suffices, ("gamma_dmpq_tdc.test_tdc_state_machine_hand_sequence",
                                   "gamma_dmpq_tdc.test_tdc_needs_two_computed_updates")),
    (tdc_apply_subtracts, ("gamma_dmpq_tdc.test_tdc_apply_identity",)),
    (qlinear_ignores_flag_int8, ("block.test_block_on_a_row_subset_with_the_full_tensor_amaxes",
                                 "delayed.test_block_converges_to_dynamic_at_fixed_input")),
    (qlinear_ignores_flag_nvfp4, ("delayed.test_int8_layers_are_unchanged_by_fusion",)),
    (dmpq_never_picks_nvfp4, ("block.test_stack_flags_follow_gamma_and_uniform_extremes",)),
    (mx_scale_exponent_one_low, ("mxcache.test_grid_values_round_trip", "mxcache.test_scale_boundary_and_powers_of_two")),
    (mx_layout_scales_first, ("mxcache.test_layout_codes_then_scales",)),
    (r_squared_complement, ("calib.test_fit_line_recovers_exact_lines", "calib.test_fit_line_hand_example")),
    (fit_line_swapped, ("calib.test_fit_line_recovers_exact_lines", "calib.test_fit_line_hand_example")),
    (cosine_without_sqrt, ("calib.test_cosine_closed_forms",)),
]


@pytest.mark.parametrize("plant,pins", MUTANTS, ids=[m[0].__name__ for m in MUTANTS])
def test_planted_mistake_is_caught_by_a_pin(monkeypatch, plant, pins):
    tests = _pins(*pins)                      # import the pin modules before patching
    plant(monkeypatch)
    caught = []
    for name, fn in tests:
        try:
            fn()
        except AssertionError:                # a pin's check failed (any other error is a broken case)
            caught.append(name)
    assert caught, f"no pin caught the planted mistake {plant.__name__}: ran {[n for n, _ in tests]}"


def test_pins_pass_on_the_unmodified_oracle():
    """The same pin tests pass when nothing is planted (so a catch above is the
    planted mistake's doing)."""
    names = sorted({n for _, pins in MUTANTS for n in pins})
    for name, fn in _pins(*names):
        fn()
