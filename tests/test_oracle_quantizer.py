"""Pins for the oracle quantizer (MicroQonv §III-A, §IV-A, §IV-B).

The strongest pin is an exact-rational brute-force quantizer written here from
the same definitions (amax, T_scale, CastE4M3 of the block scale, nearest-grid
codes) with Python Fractions, and packed with numpy reshapes -- an independent
formulation of the channel-batch-first block layout -- compared byte for byte.
Closed-form round trips, zero blocks, ties, saturation, supplied statistics
and the bits-per-element figures complete it.
"""
from fractions import Fraction

import numpy as np
import pytest

from test_oracle_formats import GRIDS, brute_round

EMAX = {"e2m1": Fraction(6), "e2m3": Fraction(15, 2), "e4m3": Fraction(448)}
SBIT = {"e2m1": 8, "e2m3": 32, "e4m3": 128}


def f32_rn(fr: Fraction) -> float:
    """Nearest float32 to an exact rational (ties to even)."""
    c = np.float32(float(fr))
    cands = [c, np.nextafter(c, np.float32(-np.inf)), np.nextafter(c, np.float32(np.inf))]
    best = min(cands, key=lambda v: (abs(Fraction(float(v)) - fr),
                                     int(np.array(v, dtype=np.float32).view(np.uint32)) & 1))
    return float(best)


def blocks_of(x: np.ndarray, role: str, layout: str) -> np.ndarray:
    """(num_blocks, 64) view of a tensor in block order, in-block [a][b] with b fastest."""
    if role == "weight":
        Co, Ci, Kh, Kw = x.shape
        t = x.transpose(2, 3, 0, 1).reshape(Kh, Kw, Co // 8, 8, Ci // 8, 8)
    else:
        if layout == "hwcn":
            x = x.transpose(3, 2, 0, 1)  # (H, W, C, N) -> (N, C, H, W)
        N, C, H, W = x.shape
        t = x.transpose(2, 3, 0, 1).reshape(H, W, N // 8, 8, C // 8, 8)
    return t.transpose(0, 1, 2, 4, 3, 5).reshape(-1, 64)


def pack(codes: np.ndarray, fmt: str) -> np.ndarray:
    codes = codes.astype(np.uint8)
    if fmt == "e2m1":
        return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8).ravel()
    if fmt == "e2m3":
        bits = ((codes[:, :, None] >> np.arange(6)) & 1).astype(np.uint8).reshape(-1, 384)
        return np.packbits(bits, axis=1, bitorder="little").ravel()
    return codes.ravel()


def brute_quantize(x: np.ndarray, fmt: str, role: str, layout: str, amax_in=None):
    x = np.asarray(x, dtype=np.float32)
    amax = max(abs(Fraction(float(v))) for v in x.ravel())
    used = Fraction(float(np.float32(amax_in))) if amax_in is not None else amax
    s_t = f32_rn(used / (EMAX[fmt] * 448))
    grid, grid8 = GRIDS[fmt], GRIDS["e4m3"]
    blks = blocks_of(x, role, layout)
    scales = np.zeros(len(blks), dtype=np.uint8)
    codes = np.zeros(blks.shape, dtype=np.uint8)
    for b, blk in enumerate(blks):
        ab = max(abs(Fraction(float(v))) for v in blk)
        sc = brute_round(grid8, ab / (EMAX[fmt] * Fraction(s_t))) if s_t > 0 else 0
        scales[b] = sc
        bs = grid8[sc]
        for i, v in enumerate(blk):
            mag = brute_round(grid, Fraction(float(v)) / (bs * Fraction(s_t))) if bs > 0 else 0
            codes[b, i] = mag | (SBIT[fmt] if np.signbit(v) else 0)
    return pack(codes, fmt), scales, s_t, float(amax)


def midpoint_tensor(fmt):
    """(8, 16, 1, 1) tensor with T_scale = 1 and a block with B_scale = 1 whose
    other elements sit exactly on, or one fp32 ulp either side of, every
    rounding midpoint of the element grid."""
    g = [float(v) for v in GRIDS[fmt]]
    mids = np.array([(g[i] + g[i + 1]) / 2 for i in range(len(g) - 1)], dtype=np.float32)
    vals = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    vals = np.concatenate([vals, -vals])[:63]
    x = np.zeros((8, 16, 1, 1), dtype=np.float32)
    x[0, 0, 0, 0] = float(EMAX[fmt]) * 448          # block 0: amax -> T_scale = 1, B_scale = 448
    blk = np.zeros(64, dtype=np.float32)
    blk[0] = float(EMAX[fmt])                        # block 1: amax = maxB_ef -> B_scale = 1
    blk[1:1 + len(vals)] = vals
    x[:, 8:, 0, 0] = blk.reshape(8, 8)
    return x


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
def test_quantizer_midpoints_match_brute_force(orc, fmt):
    x = midpoint_tensor(fmt)
    q = orc.quantize(x, fmt, "act", "nchw")
    codes, scales, s_t, _ = brute_quantize(x, fmt, "act", "nchw")
    assert s_t == 1.0 and orc.decode("e4m3", scales)[1] == 1.0
    np.testing.assert_array_equal(q["scales"], scales)
    np.testing.assert_array_equal(q["codes"], codes)


CASES = [
    ("act", "nchw", (8, 8, 2, 3)),
    ("act", "nchw", (16, 8, 1, 2)),
    ("grad", "hwcn", (2, 3, 8, 8)),
    ("weight", "oihw", (8, 16, 3, 1)),
]


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
@pytest.mark.parametrize("role,layout,shape", CASES)
def test_quantizer_matches_exact_brute_force(orc, fmt, role, layout, shape):
    rng = np.random.default_rng(hash((fmt, role, shape)) & 0xFFFF)
    x = (rng.standard_normal(shape) * 0.7).astype(np.float32)
    x.ravel()[::7] = 0.0
    x.ravel()[3] = -0.0
    q = orc.quantize(x, fmt, role, layout)
    codes, scales, s_t, amax = brute_quantize(x, fmt, role, layout)
    assert q["s_t"] == s_t and q["amax"] == amax
    np.testing.assert_array_equal(q["scales"], scales)
    np.testing.assert_array_equal(q["codes"], codes)


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
def test_quantizer_supplied_amax_matches_brute_force(orc, fmt):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((8, 8, 2, 2)).astype(np.float32)
    for factor in (2.0, 0.37):  # larger statistic, and one that forces saturation
        amax_in = float(np.float32(np.abs(x).max() * factor))
        q = orc.quantize(x, fmt, "act", "nchw", amax_in=amax_in)
        codes, scales, s_t, _ = brute_quantize(x, fmt, "act", "nchw", amax_in=amax_in)
        assert q["s_t"] == s_t
        np.testing.assert_array_equal(q["scales"], scales)
        np.testing.assert_array_equal(q["codes"], codes)


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
@pytest.mark.parametrize("j", [-7, 0, 5])
def test_lossless_round_trip(orc, fmt, j):
    """Values c * bs * 2^j with c on the element grid, bs on the E4M3 grid, each
    block holding an element of magnitude maxB_ef and one block with bs = 448,
    give T_scale = 2^j exactly, block scales bs and codes c: quantizing is the
    identity and dequantizing returns the input bit for bit."""
    rng = np.random.default_rng(100 + j)
    grid = np.array([float(v) for v in GRIDS[fmt]])
    grid8 = np.array([float(v) for v in GRIDS["e4m3"]])
    N, C, H, W = 16, 16, 2, 3
    nblk = (N // 8) * (C // 8) * H * W
    bs_idx = rng.integers(40, len(grid8), nblk)   # keep c * bs * 2^j a normal fp32
    bs_idx[nblk // 2] = len(grid8) - 1            # one block at 448
    c_idx = rng.integers(0, len(grid), (nblk, 64))
    c_idx[np.arange(nblk), rng.integers(0, 64, nblk)] = len(grid) - 1  # block amax = emax * bs
    sign = rng.integers(0, 2, (nblk, 64))
    vals = np.where(sign == 1, -1.0, 1.0) * grid[c_idx] * grid8[bs_idx][:, None] * 2.0 ** j
    # scatter blocks back to NCHW: inverse of blocks_of
    t = vals.reshape(H, W, N // 8, C // 8, 8, 8).transpose(0, 1, 2, 4, 3, 5).reshape(H, W, N, C)
    x = np.ascontiguousarray(t.transpose(2, 3, 0, 1)).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), t.transpose(2, 3, 0, 1))  # exact in fp32
    q = orc.quantize(x, fmt, "act", "nchw")
    assert q["s_t"] == 2.0 ** j
    np.testing.assert_array_equal(q["scales"], bs_idx.astype(np.uint8))
    expect_codes = (c_idx | np.where(sign == 1, SBIT[fmt], 0)).astype(np.uint8)
    np.testing.assert_array_equal(q["codes"], pack(expect_codes, fmt))
    np.testing.assert_array_equal(orc.dequantize(q), x.astype(np.float64))


def test_zero_tensor_and_zero_blocks(orc):
    x = np.zeros((8, 16, 2, 2), dtype=np.float32)
    x[:, :, 0, 0] = -0.0
    q = orc.quantize(x, "e2m1", "act", "nchw")
    assert q["s_t"] == 0.0 and q["amax"] == 0.0
    assert not q["scales"].any()
    codes = orc.unpack_codes(q)
    # sign bits follow the inputs (-0.0 at position (0, 0)); magnitudes are 0
    assert np.all((codes & 7) == 0)
    assert np.all(codes[:2] == 8) and np.all(codes[2:] == 0)
    # a nonzero tensor with one all-zero block
    x = np.ones((8, 16, 1, 1), dtype=np.float32)
    x[:, 8:, 0, 0] = 0.0
    q = orc.quantize(x, "e2m1", "act", "nchw")
    assert q["scales"][1] == 0 and q["scales"][0] != 0
    assert np.all(orc.unpack_codes(q)[1] == 0)


def test_scale_tie_rounds_to_even(orc):
        # s_t = 1 (amax = 6 * 448).  Block 1's amax 6 * 1.1875 puts its scale quotient
    # exactly halfway between E4M3 1.125 (odd code) and 1.25 (even code).
    x = np.zeros((8, 16, 1, 1), dtype=np.float32)
    x[0, 0, 0, 0] = 2688.0
    x[1, 8, 0, 0] = 6 * 1.1875
    q = orc.quantize(x, "e2m1", "act", "nchw")
    assert q["s_t"] == 1.0
    bs = orc.decode("e4m3", q["scales"])
    assert bs[0] == 448.0
    assert bs[1] == 1.25


def test_nonfinite_input_raises(orc):
    x = np.ones((8, 8, 1, 1), dtype=np.float32)
    x[3, 3, 0, 0] = np.inf
    with pytest.raises(FloatingPointError):
        orc.quantize(x, "e2m1", "act", "nchw")
    x[3, 3, 0, 0] = np.nan
    with pytest.raises(FloatingPointError):
        orc.quantize(x, "e2m1", "act", "nchw")


@pytest.mark.parametrize("fmt,bits", [("e2m1", 4.125), ("e2m3", 6.125), ("e4m3", 8.125)])
def test_bits_per_element(orc, fmt, bits):
    dims = (64, 128, 7, 7)
    sz = orc.packed_sizes(fmt, "act", dims)
    assert 8 * (sz["code_bytes"] + sz["scale_bytes"]) / np.prod(dims) == bits


def test_hwcn_equals_nchw(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((16, 24, 3, 2)).astype(np.float32)
    a = orc.quantize(x, "e2m3", "grad", "nchw")
    b = orc.quantize(np.ascontiguousarray(x.transpose(2, 3, 1, 0)), "e2m3", "grad", "hwcn")
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["scales"], b["scales"])
