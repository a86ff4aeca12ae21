"""Pins for the oracle's element formats and its rounding.

The grids are checked against an independent construction (uniform spacing
per binade, written from the format's definition of exponent and mantissa
widths) and, for E4M3, against torch's float8_e4m3fn decoding of all 256 bit
patterns.  The rounding is checked against exact rational brute force over
the whole grid and against torch's float32 -> float8_e4m3fn cast.

Formats: NVFP4 elements E2M1 with an E4M3 block scale (MicroQonv §II-D,
§III-A: maxB_sf = 448, maxB_ef = 6); the 8-bit variant uses E4M3 elements
(§IV-E) and the 6-bit variant E2M3 elements (§VI-B).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch


def spacing_grid(ebits, mbits, bias, drop_top=False):
    """Non-negative grid built binade by binade: the subnormal range [0, 2^(1-bias))
    holds 2^mbits evenly spaced values, each normal binade [2^e, 2^(e+1)) another
    2^mbits; the spacing in binade e is 2^(e - mbits)."""
    vals = []
    step = Fraction(2) ** (1 - bias - mbits)
    vals += [k * step for k in range(2 ** mbits)]
    for e in range(1 - bias, (2 ** ebits - 1) - bias + 1):
        lo = Fraction(2) ** e
        step = Fraction(2) ** (e - mbits)
        vals += [lo + k * step for k in range(2 ** mbits)]
    if drop_top:
        vals = vals[:-1]
    return vals


GRIDS = {
    "e2m1": spacing_grid(2, 1, 1),
    "e2m3": spacing_grid(2, 3, 1),
    "e4m3": spacing_grid(4, 3, 7, drop_top=True),   # S.1111.111 is NaN in E4M3 "FN"
}


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
def test_grid_matches_binade_construction(orc, fmt):
    g = orc.format_grid(fmt)
    assert [Fraction(v) for v in g] == GRIDS[fmt]


def test_grid_maxima_printed_on_pages(orc):
    # maxB_ef = 6 for FP4 E2M1 and maxB_sf = 448 for FP8 E4M3 (MicroQonv §III-A)
    assert orc.format_grid("e2m1")[-1] == 6.0
    assert orc.format_grid("e4m3")[-1] == 448.0
    assert list(orc.format_grid("e2m1")) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_decode_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    finite = ~np.isnan(ref)
    assert finite.sum() == 254
    ours = orc.decode("e4m3", codes)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    # sign handling of zero: 0x80 is -0
    assert np.signbit(ours[0x80]) and ours[0x80] == 0.0


def brute_round(grid, q: Fraction):
    """Nearest grid point by exhaustive exact search; ties to the even index;
    beyond the top value clamp to it."""
    a = abs(q)
    best = None
    for i, g in enumerate(grid):
        d = abs(a - g)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def probe_values(fmt, rng):
    g = [float(v) for v in GRIDS[fmt]]
    mids = [(g[i] + g[i + 1]) / 2 for i in range(len(g) - 1)]
    vals = [0.0, -0.0, g[-1], g[-1] * 1.01, g[-1] * 10, 1e-30]
    for m in mids:
        vals += [m, np.nextafter(m, 0.0), np.nextafter(m, np.inf)]
    vals += list(np.float32(rng.uniform(0, g[-1] * 1.1, 400)).astype(np.float64))
    vals += list(rng.uniform(0, g[1] * 4, 100))
    vals = np.array(vals, dtype=np.float64)
    return np.concatenate([vals, -vals])


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
def test_rounding_matches_exact_brute_force(orc, fmt):
    rng = np.random.default_rng(11)
    q = probe_values(fmt, rng)
    codes = orc.round_codes(fmt, q)
    sbit = {"e2m1": 8, "e2m3": 32, "e4m3": 128}[fmt]
    grid = GRIDS[fmt]
    for v, c in zip(q, codes):
        assert (c & (sbit - 1)) == brute_round(grid, Fraction(float(v))), (fmt, v, c)
        assert bool(c & sbit) == bool(np.signbit(v)), (fmt, v, c)


def test_rounding_matches_torch_e4m3_cast(orc):
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.uniform(-464, 464, 20000).astype(np.float32),
        (rng.standard_normal(20000) * 0.01).astype(np.float32),
        np.float32(2.0 ** rng.uniform(-12, 8.8, 20000)),
    ]).astype(np.float32)
    x = x[np.abs(x) < 464]  # torch maps |x| >= 464 to NaN instead of saturating
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = orc.round_codes("e4m3", x.astype(np.float64))
    np.testing.assert_array_equal(ours, ref)


def test_ties_go_to_even(orc):
    # E2M1: 0.25 -> 0 (code 0), 0.75 -> 1.0 (code 2), 1.25 -> 1.0, 1.75 -> 2.0, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    q = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert list(orc.decode("e2m1", orc.round_codes("e2m1", q))) == [0, 1, 1, 2, 2, 4, 4]


def test_saturation(orc):
    for fmt, top in (("e2m1", 6.0), ("e2m3", 7.5), ("e4m3", 448.0)):
        v = orc.decode(fmt, orc.round_codes(fmt, np.array([top * 1.5, 1e30, -1e30])))
        assert list(v) == [top, top, -top]


def test_tensor_scale_is_one_fp32_division(orc):
    rng = np.random.default_rng(5)
    for fmt, emax in (("e2m1", 6.0), ("e2m3", 7.5), ("e4m3", 448.0)):
        for a in np.float32(rng.uniform(1e-3, 1e3, 200)):
            exact = Fraction(float(a)) / Fraction(emax * 448)
            got = orc.tensor_scale(fmt, float(a))
            # fp32 RN of the exact quotient: the neighbours are farther away
            f = np.float32(got)
            lo, hi = np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(np.inf))
            assert abs(Fraction(float(f)) - exact) <= abs(Fraction(float(lo)) - exact)
            assert abs(Fraction(float(f)) - exact) <= abs(Fraction(float(hi)) - exact)
        assert orc.tensor_scale(fmt, emax * 448 * 0.5) == 0.5
        assert orc.tensor_scale(fmt, 0.0) == 0.0
