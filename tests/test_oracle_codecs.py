"""Pins of the oracle's number formats against the format definitions and
against library conversions (torch's float8_e4m3fn and bfloat16)."""
import os

import numpy as np
import pytest
import torch

from oracle import codecs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_e2m1_decode_table():
    for code, val in _rows("e2m1_table.txt"):
        got = codecs.e2m1_decode(int(code))
        assert float(got) == float(val)
        assert np.signbit(got) == val.startswith("-")


def test_e2m1_grid_round_trip():
    for code in range(16):
        v = codecs.e2m1_decode(code)
        assert int(codecs.e2m1_encode(v)) == code


def test_e2m1_rounding_fixture():
    for x, code in _rows("e2m1_rounding.txt"):
        assert int(codecs.e2m1_encode(np.float32(float(x)))) == int(code), x


def test_e2m1_nearest_brute_force():
    # every encode is a nearest grid point; among equally near points the even code
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.uniform(-7, 7, 4000), np.arange(-26, 27) * 0.25]).astype(np.float32)
    codes = codecs.e2m1_encode(x)
    grid = np.array([float(v) for _, v in _rows("e2m1_table.txt")[:8]])
    for xi, c in zip(x, codes):
        a = min(abs(float(xi)), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        expect = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert (int(c) & 7) == expect
        assert (int(c) >> 3) == int(np.signbit(xi))


def test_e2m1_pack_low_nibble_first():
    codes = np.array([[1, 2, 15, 0]], dtype=np.uint8)
    p = codecs.pack_e2m1(codes)
    assert p.tolist() == [[0x21, 0x0F]]
    assert np.array_equal(codecs.unpack_e2m1(p), codes)


def test_e4m3_decode_all_codes_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = codecs.e4m3_decode(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert float(codecs.e4m3_decode(0x7E)) == 448.0
    assert float(codecs.e4m3_decode(0x01)) == 2.0 ** -9


def test_e4m3_encode_vs_torch_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(0, 448, 20000), np.exp2(rng.uniform(-12, 8.8, 20000)).clip(0, 448),
                        codecs.e4m3_decode(np.arange(0x7F))]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codecs.e4m3_encode(x), ref)


def test_e4m3_fixture_points():
    for x, code in _rows("e4m3_points.txt"):
        assert int(codecs.e4m3_encode(np.float32(float(x)))) == int(code, 16), x


def test_bf16_vs_torch():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(50000) * np.exp2(rng.integers(-20, 20, 50000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(codecs.f32_to_bf16(x), ref)
    back = torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(codecs.bf16_to_f32(ref), back)
