"""Pins for the oracle's E4M3 codec (CPU only).

Each check ties the oracle to something other than itself: facts the pages
print (tests/golden/e4m3_format_facts.txt), brute force over all 256 codes,
every rounding midpoint of the grid, and PyTorch's own float8_e4m3fn cast
as an independent witness for values within +-448.
"""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden

FINITE = [c for c in range(256) if (c & 0x7F) != 0x7F]


def torch_decode(codes):
    t = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_encode(values_f32):
    t = torch.tensor(np.asarray(values_f32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_codes_matches_torch(oracle_mod):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle_mod.e4m3_decode(codes)
    ref = torch_decode(list(range(256)))
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            assert math.isnan(ours[c]), c
        else:
            assert ours[c] == ref[c], (hex(c), ours[c], ref[c])


def test_format_facts_from_pages(oracle_mod):
    g = read_golden("e4m3_format_facts.txt")
    c96 = int(g["bits_96"], 2)
    assert c96 == 0x6C
    assert oracle_mod.e4m3_decode([c96])[0] == 96.0
    assert oracle_mod.e4m3_encode([96.0])[0] == c96
    assert oracle_mod.e4m3_encode([95.0])[0] == oracle_mod.e4m3_encode(
        [float(g["value_95_rounds_to"])])[0]
    vals = oracle_mod.e4m3_decode(np.array(FINITE, dtype=np.uint8))
    assert np.nanmax(vals) == float(g["max_finite"]) == 448.0
    pos = sorted(v for v in vals if v > 0)
    assert pos[0] == 2.0 ** int(g["min_subnormal_log2"])
    normals = [v for c, v in zip(FINITE, vals) if v > 0 and (c >> 3) & 15]
    assert min(normals) == 2.0 ** int(g["min_normal_log2"])
    per = int(g["values_per_binade"])
    for e in range(-6, 8):          # full binades [2^e, 2^(e+1)) below 256
        n = sum(1 for v in pos if 2.0 ** e <= v < 2.0 ** (e + 1))
        assert n == per, e
    # the top binade stops at 448: the fn variant spends 0x7F on NaN
    assert sum(1 for v in pos if 256 <= v) == per - 1
    # spacing inside a binade is 1/8 of its start (12.5 %)
    b = [v for v in pos if 1.0 <= v < 2.0]
    assert np.allclose(np.diff(b), 0.125)


def test_roundtrip_every_finite_code(oracle_mod):
    vals = oracle_mod.e4m3_decode(np.array(FINITE, dtype=np.uint8))
    back = oracle_mod.e4m3_encode(vals)
    assert list(back) == FINITE
    assert oracle_mod.e4m3_encode([-0.0])[0] == 0x80
    assert oracle_mod.e4m3_encode([0.0])[0] == 0x00
    assert oracle_mod.e4m3_encode([float("nan")])[0] == 0x7F


def test_midpoints_tie_to_even_and_neighbours(oracle_mod):
    pos_codes = list(range(0x00, 0x7F))
    vals = oracle_mod.e4m3_decode(np.array(pos_codes, dtype=np.uint8))
    for sign in (1.0, -1.0):
        for i in range(len(pos_codes) - 1):
            lo, hi = vals[i], vals[i + 1]
            mid = (lo + hi) / 2.0           # exact in fp32 and fp64
            assert float(np.float32(mid)) == mid
            c_lo, c_hi = pos_codes[i], pos_codes[i + 1]
            even = c_lo if c_lo % 2 == 0 else c_hi
            sb = 0x80 if sign < 0 else 0
            got = oracle_mod.e4m3_encode([sign * mid])[0]
            assert got == (even | sb), (sign * mid, hex(got))
            up = float(np.nextafter(np.float32(mid), np.float32(np.inf)))
            dn = float(np.nextafter(np.float32(mid), np.float32(0)))
            assert oracle_mod.e4m3_encode([sign * up])[0] == (c_hi | sb)
            assert oracle_mod.e4m3_encode([sign * dn])[0] == (c_lo | sb)


def test_saturation_and_small_values(oracle_mod):
    g = read_golden("e4m3_format_facts.txt")
    for v in (448.0, 449.0, 463.99, 464.0, 480.0, 672.0, 1e9, 3.0e38):
        assert oracle_mod.e4m3_encode([v])[0] == 0x7E
        assert oracle_mod.e4m3_encode([-v])[0] == 0xFE
    # with scale 1.0: 0.001 rounds up to 2^-9; half of 2^-9 ties down to 0
    assert oracle_mod.round_e4m3([0.001])[0] == 2.0 ** int(
        g["kv_scale1_0.001_rounds_to_log2"])
    assert oracle_mod.e4m3_encode([0.001])[0] == 0x01
    assert oracle_mod.e4m3_encode([2.0 ** -10])[0] == 0x00
    assert oracle_mod.e4m3_encode([float(np.nextafter(np.float32(2 ** -10),
                                                      np.float32(1)))])[0] == 0x01
    assert oracle_mod.e4m3_encode([3 * 2.0 ** -10])[0] == 0x02
    assert oracle_mod.e4m3_encode([-1e-5])[0] == 0x80


def test_encode_matches_torch_cast_within_range(oracle_mod):
    rng = np.random.default_rng(12345)
    n = 60000
    mag = np.exp2(rng.uniform(-12.0, math.log2(448.0), n))
    v = (mag * np.where(rng.random(n) < 0.5, -1.0, 1.0)).astype(np.float32)
    ours = oracle_mod.e4m3_encode(v.astype(np.float64))
    ref = torch_encode(v)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:5]]


def test_round_e4m3_is_decode_of_encode(oracle_mod):
    rng = np.random.default_rng(7)
    v = rng.standard_normal(5000) * 50.0
    r = oracle_mod.round_e4m3(v)
    d = oracle_mod.e4m3_decode(oracle_mod.e4m3_encode(v))
    assert np.array_equal(r, d)
    # nearest grid value: no finite code is strictly closer
    grid = oracle_mod.e4m3_decode(np.array(FINITE, dtype=np.uint8))
    for x, rx in zip(v[:500], r[:500]):
        xc = max(min(x, 448.0), -448.0)
        assert abs(rx - xc) <= np.min(np.abs(grid - xc)) + 0.0


@pytest.mark.parametrize("code", [0x38, 0x39, 0x01, 0x08, 0x7E, 0xB8, 0xFE])
def test_known_codes(oracle_mod, code):
    expect = {0x38: 1.0, 0x39: 1.125, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6,
              0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}[code]
    assert oracle_mod.e4m3_decode([code])[0] == expect


def stepwise_round(x: float) -> float:
    """The rounding as the pages state it step by step ("FP8 Inference
    Explained, in depth", "The numbers in one byte"): keep the sign, clip
    the magnitude at 448, find its binade 2^e with e no lower than -6 (the
    smallest normal exponent; below it the spacing stays 2^-9), snap to the
    binade's grid of spacing 2^(e-3) with halfway cases to even, clip again.
    Written independently of the oracle, which instead picks the nearest
    entry of the decoded code table; the two must agree everywhere."""
    if x == 0.0 or math.isnan(x):
        return x
    a = min(abs(x), 448.0)
    e = max(math.frexp(a)[1] - 1, -6)
    step = 2.0 ** (e - 3)
    r = min(round(a / step) * step, 448.0)   # Python's round: half to even
    return math.copysign(r, x)


def test_table_rounding_equals_stepwise_rounding(oracle_mod):
    grid = oracle_mod.e4m3_decode(np.array(list(range(0x7F)), dtype=np.uint8))
    pts = list(grid)
    for lo, hi in zip(grid[:-1], grid[1:]):
        mid = (lo + hi) / 2.0
        pts += [mid, float(np.nextafter(mid, 0.0)), float(np.nextafter(mid, np.inf)),
                lo + (hi - lo) / 4.0, hi - (hi - lo) / 8.0]
    rng = np.random.default_rng(99)
    pts += list(np.exp2(rng.uniform(-20.0, 12.0, 20000)))
    pts += [2.0 ** -10, 3 * 2.0 ** -10, 1e-30, 447.9, 448.0, 455.99, 456.0, 464.0, 1e6]
    vals = np.array(pts + [-p for p in pts], dtype=np.float64)
    ours = oracle_mod.round_e4m3(vals)
    ref = np.array([stepwise_round(float(v)) for v in vals])
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(vals[i], ours[i], ref[i]) for i in bad[:5]]
    assert np.array_equal(np.signbit(ours), np.signbit(ref))
