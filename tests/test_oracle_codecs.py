"""Pins for the oracle's bf16 and E4M3 codecs (CPU only).

Each codec is checked against (a) hand-worked roundings in ``tests/golden``,
(b) brute-force nearest-value search over every representable value
(``tests/brute.py``, exact fractions), and (c) torch's own casts as a library
cross-check on in-range values.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import brute
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split("|")]


# --------------------------------------------------------------------- E4M3
def test_e4m3_golden_roundings():
    for val, code, _why in _rows("e4m3_rounding.txt"):
        got = int(oracle.e4m3_encode(np.array([float(val)]))[0])
        assert got == int(code, 16), (val, hex(got), code)


def test_e4m3_decode_all_codes_against_field_definition():
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.e4m3_decode(codes)
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            assert np.isnan(dec[c])
        else:
            assert Fraction(float(dec[c])) == brute.e4m3_value(c), hex(c)


def test_e4m3_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    again = oracle.e4m3_encode(oracle.e4m3_decode(codes))
    np.testing.assert_array_equal(again, codes)
    assert len(codes) == 254


def test_e4m3_largest_finite_and_saturation():
    assert oracle.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0
    assert oracle.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0 ** -9
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38], dtype=np.float64)
    np.testing.assert_array_equal(oracle.e4m3_encode(big), np.full(7, 0x7E, np.uint8))
    np.testing.assert_array_equal(oracle.e4m3_encode(-big), np.full(7, 0xFE, np.uint8))


def test_e4m3_encode_matches_brute_force_nearest():
    rng = np.random.default_rng(1)
    # every midpoint between neighbours, plus random values over the whole range
    pos = np.sort(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = (pos[1:] + pos[:-1]) / 2
    vals = np.concatenate([mids, mids * (1 + 1e-9), mids * (1 - 1e-9),
                           rng.uniform(0, 480, 300), np.exp(rng.uniform(-14, 6, 300))])
    vals = np.concatenate([vals, -vals[::7]]).astype(np.float32).astype(np.float64)
    got = oracle.e4m3_encode(vals)
    for v, g in zip(vals, got):
        assert int(g) == brute.round_e4m3_satfinite(Fraction(float(v))), (v, hex(int(g)))


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(3)
    v = (torch.randn(200_000, generator=g) * torch.exp(torch.randn(200_000, generator=g) * 3))
    v = v.clamp(-448, 448)
    ref = v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(v.numpy().astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    dec_ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(dec_ref))
    ok = ~np.isnan(dec)
    np.testing.assert_array_equal(dec[ok], dec_ref[ok])


def test_e4m3_scaled_int_is_integer_and_bounded():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    s = oracle.e4m3_to_scaled_int(codes)
    assert np.all(s == np.round(s))
    assert np.max(np.abs(s)) == 229376


# --------------------------------------------------------------------- bf16
def test_bf16_golden_roundings():
    for val, bits, _why in _rows("bf16_rounding.txt"):
        got = int(oracle.f64_to_bf16(np.array([float(val)]))[0])
        assert got == int(bits, 16), (val, hex(got), bits)


def test_bf16_matches_torch_cast_on_random_f32():
    g = torch.Generator().manual_seed(5)
    n = 1 << 20
    v = torch.randn(n, generator=g) * torch.exp(torch.randn(n, generator=g) * 20)
    # also exact-tie patterns: random fp32 bit patterns with the low 16 bits = 0x8000
    ties = (torch.randint(0, 1 << 15, (1 << 16,), generator=g, dtype=torch.int32) << 16) | 0x8000
    tiesf = ties.view(torch.float32)
    tiesf = tiesf[torch.isfinite(tiesf)]
    v = torch.cat([v, tiesf, -tiesf])
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f32_to_bf16(v.numpy())
    np.testing.assert_array_equal(got, ref)


def test_bf16_single_rounding_from_f64_matches_brute_force():
    rng = np.random.default_rng(7)
    vals = np.concatenate([rng.standard_normal(300) * 10.0 ** rng.integers(-6, 6, 300),
                           np.array([2.0 ** -130, 3 * 2.0 ** -134, 1e-39, -5e-41])])
    got = oracle.f64_to_bf16(vals)
    for v, gbits in zip(vals, got):
        assert int(gbits) == brute.round_bf16(Fraction(float(v))), v


def test_bf16_decode_round_trip_all_finite():
    bits = np.array([b for b in range(65536) if ((b >> 7) & 0xFF) != 0xFF], dtype=np.uint16)
    np.testing.assert_array_equal(oracle.f64_to_bf16(oracle.bf16_to_f64(bits)), bits)
