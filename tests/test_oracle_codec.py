"""Pins for the oracle's E4M3 codec and bf16 rounding.

Nothing here re-types the oracle's formulas: the codec is checked against the
format's published table, an independent library (ml_dtypes / torch float8),
a second algorithm (exhaustive nearest search), and exact midpoint arithmetic.
"""
import os

import ml_dtypes
import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ocp_table.txt")


def _finite_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_decode_matches_ocp_table(orc):
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 10
    for code_hex, val in rows:
        got = orc.e4m3_decode([int(code_hex, 16)])[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val) and np.signbit(got) == val.startswith("-")


def test_decode_all_codes_match_ml_dtypes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    got = orc.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))


def test_decode_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_decode(np.arange(256))
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[fin], ref[fin])


def test_roundtrip_every_code(orc):
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.e4m3_decode(codes).astype(np.float32)
    back = orc.e4m3_encode(vals)
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            assert back[c] == 0x7F  # NaN -> canonical NaN
        else:
            assert back[c] == c, hex(c)


def test_midpoints_tie_to_even_and_neighbours(orc):
    pos = [c for c in _finite_codes() if c < 0x80]
    vals = orc.e4m3_decode(pos)
    for i in range(len(pos) - 1):
        lo, hi = vals[i], vals[i + 1]
        mid = np.float32((lo + hi) / 2)  # exact: <= 5 significant bits
        assert float(mid) == (lo + hi) / 2
        even = pos[i] if pos[i] % 2 == 0 else pos[i + 1]
        for sgn, sbit in ((1, 0), (-1, 0x80)):
            assert orc.e4m3_encode([sgn * mid])[0] == even | sbit
            below = np.nextafter(mid, np.float32(0), dtype=np.float32)
            above = np.nextafter(mid, np.float32(np.inf), dtype=np.float32)
            assert orc.e4m3_encode([sgn * below])[0] == pos[i] | sbit
            assert orc.e4m3_encode([sgn * above])[0] == pos[i + 1] | sbit


def test_saturation_and_specials(orc):
    cases = [
        (448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (464.0001, 0x7E), (479.9, 0x7E),
        (480.0, 0x7E), (1e30, 0x7E), (np.inf, 0x7E), (-np.inf, 0xFE), (-1e30, 0xFE),
        (-464.0, 0xFE), (0.0, 0x00), (-0.0, 0x80),
        (2.0 ** -10, 0x00),                     # tie between 0 and 2^-9 -> even (0)
        (2.0 ** -10 * (1 + 2.0 ** -23), 0x01),
        (-(2.0 ** -10) * (1 + 2.0 ** -23), 0x81),
        (3 * 2.0 ** -10, 0x02),                 # tie between codes 1 and 2 -> even
        (2.0 ** -9, 0x01), (2.0 ** -6, 0x08), (1.0, 0x38), (1e-30, 0x00), (-1e-30, 0x80),
        (1e-40, 0x00),                          # fp32 subnormal input
    ]
    vals = np.array([c[0] for c in cases], dtype=np.float32)
    got = orc.e4m3_encode(vals)
    for v, g, want in zip(vals, got, [c[1] for c in cases]):
        assert g == want, (float(v), hex(g), hex(want))
    assert orc.e4m3_encode([np.float32(np.nan)])[0] == 0x7F


def _probe_values():
    rng = np.random.default_rng(123)
    allbf = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    rnd = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    inrange = (rng.uniform(-500, 500, size=200_000)).astype(np.float32)
    small = (rng.uniform(-2 ** -5, 2 ** -5, size=100_000)).astype(np.float32)
    v = np.concatenate([allbf, rnd, inrange, small])
    return v[~np.isnan(v)]


def test_arithmetic_encoder_matches_nearest_search(orc):
    v = _probe_values()
    a = orc.e4m3_encode(v)
    b = orc.e4m3_encode_search(v)
    bad = np.nonzero(a != b)[0]
    assert bad.size == 0, [(float(v[i]), hex(a[i]), hex(b[i])) for i in bad[:5]]


def test_encoder_matches_ml_dtypes_in_range(orc):
    v = _probe_values()
    v = v[np.abs(v) <= 448]
    ref = v.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    got = orc.e4m3_encode(v)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_encoder_matches_torch_in_range(orc):
    v = _probe_values()
    v = v[np.abs(v) <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(v), ref)


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.integers(0, 2 ** 32, size=20_000, dtype=np.uint64).astype(np.uint32).view(np.float32),
        # exact ties: low 16 bits = 0x8000 with both parities of bit 16
        ((rng.integers(0, 2 ** 16, size=2000, dtype=np.uint32) << 16) | 0x8000).view(np.float32),
    ])
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_rne(v), ref)
