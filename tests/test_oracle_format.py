"""Pins of the CPU oracle's scalar formats (E2M1, E4M3, BF16, FP16, FP32 roundings).

Each check ties the oracle to something other than itself: the grid and anchor values printed
in golden fixtures (with their sources), a brute-force nearest-value search over the grid, or an
independent library conversion (numpy / torch casts)."""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


def _grid():
    return {int(c): float(v) for c, v in read_golden("e2m1_grid.txt")}


def brute_e2m1(y: float) -> int:
    """Nearest E2M1 code by exhaustive search over the 8 magnitudes (exact rationals), ties to
    the even code, magnitudes above 6 saturated, sign bit from the sign of y."""
    grid = _grid()
    mags = [(Fraction(grid[c]), c) for c in range(8)]
    a = Fraction(abs(y))
    if a >= 6:
        best = 7
    else:
        dist = [(abs(a - m), c) for m, c in mags]
        dmin = min(d for d, _ in dist)
        cands = [c for d, c in dist if d == dmin]
        best = min(cands, key=lambda c: (c & 1, c))
    sign = 8 if math.copysign(1.0, y) < 0 else 0
    return sign | best


def test_e2m1_grid_matches_golden():
    grid = _grid()
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert v == grid[code] and math.copysign(1, v) == math.copysign(1, grid[code])


def test_e2m1_ties_golden():
    for x, code in read_golden("e2m1_ties.txt"):
        assert oracle.e2m1_encode(float(x)) == int(code), x


def test_e2m1_rounding_brute_force():
    rng = np.random.default_rng(1)
    xs = [k / 64.0 for k in range(-8 * 64, 8 * 64 + 1)]           # dense lattice incl. ties
    xs += list(rng.uniform(-10, 10, 2000)) + list(rng.normal(0, 1e-3, 200))
    grid = sorted(set(abs(v) for v in _grid().values()))
    for i in range(len(grid) - 1):                                  # midpoints and neighbours
        mid = (grid[i] + grid[i + 1]) / 2
        for m in (mid, np.nextafter(mid, 0), np.nextafter(mid, 10)):
            xs += [float(m), -float(m)]
    xs += [0.0, -0.0, 6.0, 6.5, 7.0, 1e30, -1e30, 5e-324, -5e-324]
    xs = [float(np.float32(x)) for x in xs]
    for x in xs:
        assert oracle.e2m1_encode(x) == brute_e2m1(x), x


def test_e4m3_values_golden_and_torch():
    for b, v in read_golden("e4m3_values.txt"):
        got = oracle.e4m3_value(int(b, 16))
        assert got == float(v) and math.copysign(1, got) == math.copysign(1, float(v))
    # every byte against torch's float8_e4m3fn decoding (library routine)
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    for b in range(256):
        got, want = oracle.e4m3_value(b), ref[b].item()
        if math.isnan(want):
            assert math.isnan(got) and (b & 0x7F) == 0x7F
        else:
            assert got == want, hex(b)


def test_e4m3_encode_against_torch():
    """RNE to E4M3 versus torch's fp32 -> float8_e4m3fn cast, on values below the overflow
    threshold (torch turns >= 464 into NaN; the format here saturates, checked separately)."""
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.uniform(-460, 460, 20000), rng.normal(0, 1, 20000),
        rng.normal(0, 1e-2, 5000), rng.uniform(-2e-3, 2e-3, 5000),
        # every E4M3 value, midpoint and neighbour
        np.array([oracle.e4m3_value(b) for b in range(0x7F)]),
    ]).astype(np.float32)
    allv = np.array(sorted(oracle.e4m3_value(b) for b in range(0x7F)))
    mids = ((allv[1:] + allv[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e3)])
    vals = vals[np.abs(vals) < 464].astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_f32(vals)
    # torch maps a value rounding to zero to +0/-0 by sign like the format; compare bytes
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_e4m3_saturation():
    for x in (464.0, 480.0, 1e4, 3e38):
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00      # tie between 0 and 2^-9 -> even (0)
    assert oracle.e4m3_encode(1.5 * 2.0 ** -9) == 0x02  # tie between 1 and 2 (x 2^-9) -> 2


def test_fp32_bf16_fp16_roundings_against_library_casts():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-30, 300),
                        rng.normal(0, 1e30, 300), rng.uniform(-7e4, 7e4, 3000)])
    for v in x:
        assert oracle.fp32(float(v)) == float(np.float32(v))
    x32 = x.astype(np.float32)
    bf = torch.from_numpy(x32).to(torch.bfloat16).float().numpy()
    for v, want in zip(x32, bf):
        assert oracle.bf16_round(float(v)) == float(want)
    h = x.astype(np.float16)  # numpy double -> half is correctly rounded
    for v, want in zip(x, h):
        got = oracle.fp16_round(float(v))
        assert got == float(want) or (math.isinf(got) and math.isinf(float(want)))


def test_bit_pattern_codecs_roundtrip():
    for hbits in range(0, 65536, 7):
        v = oracle.bf16_value(hbits)
        if math.isfinite(v):
            assert oracle.bf16_bits(v) == hbits
            assert struct.unpack("<f", struct.pack("<I", hbits << 16))[0] == v or math.isnan(v)
        v = oracle.fp16_value(hbits)
        if math.isfinite(v):
            assert oracle.fp16_bits(v) == hbits
            assert float(np.array([hbits], np.uint16).view(np.float16)[0]) == v


def test_round_to_format_definition_points():
    # E2M1 as a 2-bit-significand format with emin 0: subnormal step 0.5
    assert [oracle.round_to_format(v, 2, 0) for v in (0.2, 0.3, 0.74, 0.76, 2.6)] == \
        [0.0, 0.5, 0.5, 1.0, 3.0]
    # E4M3 subnormal grid: multiples of 2^-9 below 2^-6
    assert oracle.round_to_format(3.4 * 2 ** -9, 4, -6) == 3 * 2 ** -9
