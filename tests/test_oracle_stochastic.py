"""Pins for the oracle's stochastic rounding of element codes (MicroQonv
§III-A: Round is round-to-nearest or stochastic; stochastic for gradients).

  * the random source reproduces the published Philox4x32-10 known answers;
  * every code is one of the two grid values around the exact real quotient
    x / (B_scale T_scale) (or the largest one, saturating), values on the grid
    keep their code, and the block scales are the round-to-nearest ones;
  * over many seeds the dequantized value is unbiased: its mean converges to
    x within the binomial standard error;
  * one seed gives one result; different seeds give different codes.
"""
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
FMTS = ["e2m1", "e2m3", "e4m3"]


def test_philox_known_answers(orc):
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        np.testing.assert_array_equal(orc.philox4x32_10(v[0:4], v[4:6]), np.array(v[6:10], dtype=np.uint32))


def _exact_quotients(orc, x, q):
    """|x| / (B_scale T_scale) per element in packed order, in fp64 (exact
    enough: see the oracle header), with the block of each element."""
    N, C, H, W = q["dims"]
    bs = orc.decode("e4m3", q["scales"])
    blk = np.arange(bs.size).repeat(64)
    i = np.tile(np.arange(64), bs.size)
    pos, rest = np.divmod(blk, (N // 8) * (C // 8))
    ng, cg = np.divmod(rest, C // 8)
    h, w = np.divmod(pos, W)
    n, c = ng * 8 + i // 8, cg * 8 + i % 8
    xv = x[n, c, h, w].astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = np.where(bs[blk] > 0, np.abs(xv) / (bs[blk] * q["s_t"]), 0.0)
    return quot, xv, bs[blk]


@pytest.mark.parametrize("fmt", FMTS)
def test_codes_are_grid_neighbours_of_the_exact_quotient(orc, fmt):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((16, 16, 5, 6)) * np.exp(rng.uniform(-4, 4, (16, 16, 5, 6)))).astype(np.float32)
    x.ravel()[::9] = 0.0
    rn = orc.quantize(x, fmt, "grad", "nchw")
    sr = orc.quantize(x, fmt, "grad", "nchw", sr_seed=12345)
    np.testing.assert_array_equal(sr["scales"], rn["scales"])       # block scales stay round-to-nearest
    assert sr["s_t"] == rn["s_t"]
    grid = orc.format_grid(fmt)
    quot, xv, _ = _exact_quotients(orc, x, sr)
    mbits = {"e2m1": 3, "e2m3": 5, "e4m3": 7}[fmt]           # magnitude bits below the sign bit
    mags = grid[orc.unpack_codes(sr).ravel() & ((1 << mbits) - 1)]
    lo_idx = np.clip(np.searchsorted(grid, quot, side="right") - 1, 0, len(grid) - 1)
    lo = grid[lo_idx]
    hi = grid[np.minimum(lo_idx + 1, len(grid) - 1)]
    sat = quot >= grid[-1]
    on_grid = grid[lo_idx] == quot
    assert np.all(np.where(sat, mags == grid[-1], (mags == lo) | (mags == hi)))
    assert np.all(mags[on_grid & ~sat] == quot[on_grid & ~sat])
    assert np.any((mags != grid[np.abs(grid[None, :] - quot[:, None]).argmin(axis=1)]) & ~sat)   # not RN


@pytest.mark.parametrize("fmt", FMTS)
def test_unbiased_over_seeds(orc, fmt):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((8, 8, 2, 2)).astype(np.float32)
    rn = orc.quantize(x, fmt, "grad", "nchw")
    grid = orc.format_grid(fmt)
    quot, xv, bsv = _exact_quotients(orc, x, rn)
    mbits = {"e2m1": 3, "e2m3": 5, "e4m3": 7}[fmt]
    seeds = 800
    acc = np.zeros(quot.size)
    for s in range(seeds):
        q = orc.quantize(x, fmt, "grad", "nchw", sr_seed=1000003 * s + 7)
        acc += grid[orc.unpack_codes(q).ravel() & ((1 << mbits) - 1)]
    mean = acc / seeds
    lo_idx = np.clip(np.searchsorted(grid, quot, side="right") - 1, 0, len(grid) - 2)
    spacing = grid[lo_idx + 1] - grid[lo_idx]
    f = (quot - grid[lo_idx]) / spacing
    se = spacing * np.sqrt(np.maximum(f * (1 - f), 1e-12) / seeds)
    ok = quot < grid[-1]
    z = np.abs(mean - quot)[ok] / se[ok]
    assert np.max(z) < 5.5, f"worst deviation {np.max(z):.2f} standard errors"
    assert abs(np.mean((mean - quot)[ok] / spacing[ok])) < 0.01


def test_seed_determinism(orc):
    x = np.random.default_rng(1).standard_normal((16, 8, 3, 3)).astype(np.float32)
    a = orc.quantize(x, "e2m1", "grad", "nchw", sr_seed=99)
    b = orc.quantize(x, "e2m1", "grad", "nchw", sr_seed=99)
    c = orc.quantize(x, "e2m1", "grad", "nchw", sr_seed=100)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    assert not np.array_equal(a["codes"], c["codes"])
