"""Pins from the figures the pages print: Table I's quantization counts and
backward memory movement, the storage ratios, and the property MicroQonv is
built on -- every im2col copy of an activation, gathered from the packed
channel-batch-first tensor, carries the identical code and scale, whereas
quantizing after im2col gives copies of one activation different values
(MicroQonv §III-C, §IV-A, §IV-C, Table I; news summary of the preprint).
"""
import os

import numpy as np
import pytest

import synthetic as S
from synthetic import Layer

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_table(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            parts = line.split()
            rows[parts[0]] = [float(v) for v in parts[1:]]
    return rows


LAYER = Layer(8, 16, 8, 8, 16, 3, 1, 1)   # 3x3, stride 1, padding 1 (Table I setting)


@pytest.mark.parametrize("flow", ["dacapo", "cuyckens", "microqonv"])
def test_table1_quantization_counts(orc, flow):
    q_a, q_w, q_g, _, _ = read_table("table1_quantization_counts.txt")[flow]
    c = orc.flow_quantization_counts(LAYER, flow)
    X = c["X"].reshape(LAYER.x_shape())
    interior = X[:, :, 1:-1, 1:-1]
    assert np.all(interior == q_a)
    assert np.all(X >= 1) and np.all(X <= q_a)
    assert np.all(c["W"] == q_w)
    assert np.all(c["G"] == q_g)


def test_table1_backward_movement(orc):
    table = read_table("table1_quantization_counts.txt")
    base = orc.backward_storage_bits(LAYER, "microqonv", 4, 16)
    # 7.53 = 32 / 4.25: a 16-bit slot per 64-element block (see storage test below)
    assert round(orc.backward_storage_bits(LAYER, "dacapo", 4, 16) / base, 2) == table["dacapo"][3]
    # the im2col-expanded tensor is Kh*Kw = 9 times larger at stride 1, padding 1
    assert orc.backward_storage_bits(LAYER, "cuyckens", 4, 16) / base == table["cuyckens"][3]
    assert orc.backward_storage_bits(LAYER, "cuyckens", 4, 8) / orc.backward_storage_bits(
        LAYER, "microqonv", 4, 8) == table["cuyckens"][3]


def test_storage_ratios(orc):
    g = {k: v[0] for k, v in read_table("storage_ratios.txt").items()}
    dims = (64, 64, 8, 8)
    n = np.prod(dims)

    def packed_bits(fmt):
        sz = orc.packed_sizes(fmt, "act", dims)
        return 8.0 * (sz["code_bytes"] + sz["scale_bytes"]) / n

    b4, b6, b8 = packed_bits("e2m1"), packed_bits("e2m3"), packed_bits("e4m3")
    assert (b4, b6, b8) == (4.125, 6.125, 8.125)
    # With the 8-bit E4M3 block scale the FP4 ratio is 7.76: "up to x7.53" holds.
    assert 32.0 / b4 >= g["fp4_vs_fp32_up_to"]
    # x7.53 itself and x5.1 correspond to 16 bits of scale storage per block ...
    assert round(32.0 / (4 + 16 / 64), 2) == g["fp4_vs_fp32_up_to"]
    assert round(32.0 / (6 + 16 / 64), 1) == g["fp6_plus_vs_dacapo"]
    assert round(9 * (4 + 16 / 64) / (6 + 16 / 64)) == g["fp6_plus_vs_cuyckens"]
    assert round(9 * b4 / b6) == g["fp6_plus_vs_cuyckens"]
    # ... while x3.93 and 3.125 bits correspond to the 8-bit scale this format stores.
    assert np.floor(100 * 32.0 / b8) / 100 == g["fp8_vs_fp32"]
    assert 3 + 8 / 64 == g["unsigned_fp4_bits"]


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
def test_im2col_copies_identical_from_packed(orc, fmt):
    wl = S.WORKLOADS[0]
    X = S.draw_x(wl, 0)
    q = orc.quantize(X, fmt, "act", "nchw")
    vals, codes, scales = orc.gather_im2col_from_packed(q, LAYER)
    idx = orc.im2col_index(LAYER)
    deq = orc.dequantize(q).ravel()
    valid = idx >= 0
    # every copy carries its source element's one code, one scale, one value
    src_codes = orc.unpack_codes(q)
    for e in np.unique(idx[valid])[::37]:
        m = idx == e
        assert len(set(codes[m].tolist())) == 1
        assert len(set(scales[m].tolist())) == 1
        assert np.all(vals[m] == deq[e])
    assert np.all(codes[valid] >= 0) and src_codes.shape[1] == 64


def test_quantize_after_im2col_gives_copies_different_values(orc):
    wl = S.WORKLOADS[0]
    X = S.draw_x(wl, 0)
    Q, idx = orc.flow_quantize_after_im2col(X, LAYER, "e2m1")
    valid = idx >= 0
    differing = 0
    for e in np.unique(idx[valid]):
        v = Q[idx == e]
        if np.ptp(v) > 0:
            differing += 1
    assert differing > 0.25 * np.unique(idx[valid]).size


def test_codes_and_scales_stay_finite(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((16, 16, 3, 3)) * 1e3).astype(np.float32)
    for fmt in ("e2m1", "e2m3", "e4m3"):
        q = orc.quantize(x, fmt, "act", "nchw")
        assert np.all(q["scales"] < 0x7F)             # positive, never NaN
        if fmt == "e4m3":
            assert not np.any((orc.unpack_codes(q) & 0x7F) == 0x7F)
        assert np.all(np.isfinite(orc.dequantize(q)))


def test_square_blocks_of_cbf_im2col_are_microqonv_blocks(orc):
    """On the channel-batch-first X' every 8x8 square covers 8 channels x 8
    batch entries of one input position -- one MicroQonv block -- so squaring
    X' after that im2col reproduces quantizing X before it (the reason the
    layout lets X be quantized once, MicroQonv §IV-A/§IV-B)."""
    X = S.draw_x(S.WORKLOADS[0], 0)
    q = orc.quantize(X, "e2m1", "act", "nchw")
    vals, _, _ = orc.gather_im2col_from_packed(q, LAYER)
    idx = orc.im2col_index(LAYER, "cbf")
    M = np.where(idx >= 0, X.astype(np.float64).ravel()[np.maximum(idx, 0)], 0.0)
    np.testing.assert_array_equal(orc._fake_quantize_blocks(M, "e2m1", 8, 8), vals)


def _line_block_matrix(fmt, rows, cols, br, bc, seed):
    """A matrix whose br x bc blocks each hold grid values c * 448 * 2^(j - k)
    (k = 0..3 varying from block to block) and one element of magnitude
    maxB_ef * 448 * 2^(j - k).  With T_scale = 2^j (the largest block has
    k = 0) every block's scale is 448 * 2^-k exactly and every code is c, so
    fake quantization in exactly these blocks returns the matrix unchanged;
    in blocks of another shape the block amax mixes different k, the small
    values lose bits and the round trip breaks."""
    import oracle
    grid = oracle.format_grid(fmt)
    emax, j = grid[-1], -3
    rng = np.random.default_rng(seed)
    M = np.zeros((rows, cols))
    for b, (r0, c0) in enumerate((r, c) for r in range(0, rows, br) for c in range(0, cols, bc)):
        k = (b * 7 + 1) % 4 if b else 0
        h, w = min(br, rows - r0), min(bc, cols - c0)     # partial blocks at ragged edges
        vals = rng.choice(grid, size=(h, w)) * rng.choice([-1.0, 1.0], size=(h, w))
        vals.flat[rng.integers(h * w)] = emax
        M[r0:r0 + h, c0:c0 + w] = vals * 448.0 * 2.0 ** (j - k)
    return M


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
@pytest.mark.parametrize("br,bc", [(64, 1), (1, 64), (8, 8)])
@pytest.mark.parametrize("rows,cols", [(128, 128), (100, 72)], ids=["whole-blocks", "ragged"])
def test_line_block_round_trip(orc, fmt, br, bc, rows, cols):
    """DaCapo's line blocks of 64 along either GEMM direction (MicroQonv
    §III-C) and the 8x8 squares: lossless round trip in the right blocks
    (partial ones at ragged edges included), lossy in the transposed ones."""
    M = _line_block_matrix(fmt, rows, cols, br, bc, 7 + br)
    np.testing.assert_array_equal(orc._fake_quantize_blocks(M, fmt, br, bc), M)
    if br != bc:
        assert not np.array_equal(orc._fake_quantize_blocks(M, fmt, bc, br), M)


def test_dacapo_flow_blocks_follow_each_gemm_direction(orc):
    """flow_dacapo quantizes X' = im2col(X) twice from full precision: along
    K (its rows, 64-line blocks in a column) for the forward GEMM and along
    the (N Ho Wo) axis (64-line blocks in a row) for the weight gradient
    (MicroQonv §III-C).  A constant activation tensor on the grid round-trips
    exactly in both (every line block holds the constant or padding zeros);
    with random activations both are valid fake quantizations of X' whose
    copies of one activation differ between the two directions."""
    L = Layer(8, 64, 8, 8, 16, 3, 1, 1)       # K = 576, Ho Wo N = 512
    X = np.full(L.x_shape(), 1.5 * 448 * 2.0 ** -4, dtype=np.float32)
    Qf, Qb, idx = orc.flow_dacapo(X, L, "e2m1")
    M = np.where(idx >= 0, X.astype(np.float64).ravel()[np.maximum(idx, 0)], 0.0)
    np.testing.assert_array_equal(Qf, M)
    np.testing.assert_array_equal(Qb, M)
    X = S.draw_x(S.WORKLOADS[0], 0, L.x_shape())
    Qf, Qb, idx = orc.flow_dacapo(X, L, "e2m1")
    M = np.where(idx >= 0, X.astype(np.float64).ravel()[np.maximum(idx, 0)], 0.0)
    assert Qf.shape == Qb.shape == M.shape == (576, 512)
    assert np.all((idx >= 0) | (Qf == 0)) and np.all((idx >= 0) | (Qb == 0))
    # the two directions agree with 64-line blocks computed column by column / row by row
    np.testing.assert_array_equal(Qf[:, :1], orc._fake_quantize_blocks(M, "e2m1", 64, 1)[:, :1])
    rel_f = np.abs(Qf - M).sum() / np.abs(M).sum()
    rel_b = np.abs(Qb - M).sum() / np.abs(M).sum()
    assert 0 < rel_f < 0.2 and 0 < rel_b < 0.2
    assert not np.array_equal(Qf, Qb)
