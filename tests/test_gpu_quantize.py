"""GPU parity of mqconv_quantize_cbf: codes, scales and T_scale bit-exact
against the oracle (MicroQonv §III-A, §IV-B), for every format, source layout
and dtype, both statistic modes, edge cases, and the full-size tensors of the
workloads."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from mqtest import assert_packed_equal, gpu_quantize, to_dev

pytestmark = pytest.mark.gpu
FMTS = ["e2m1", "e2m3", "e4m3"]


def rand(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(8, 16, 8, 8), (16, 24, 7, 5), (64, 32, 3, 9), (8, 8, 1, 1),
                                   (16, 64, 5, 8), (24, 40, 4, 6), (8, 24, 2, 4), (16, 136, 6, 12)])
def test_nchw(cuda_device, fmt, dtype, shape):
    x = rand(shape, sum(shape))
    if dtype == "bf16":
        x = S.to_bf16_rne(x)
    x.ravel()[::5] = 0.0
    x.ravel()[1::7] = -0.0
    p, amax = gpu_quantize(to_dev(x, dtype, cuda_device), fmt, "act", "nchw", shape)
    ref = oracle.quantize(x, fmt, "act", "nchw")
    assert amax == ref["amax"]
    assert_packed_equal(p, ref, f"nchw {fmt} {dtype} {shape}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 3, 16, 8), (5, 4, 24, 32), (1, 1, 8, 64)])
def test_hwcn(cuda_device, fmt, dtype, shape):
    x = rand(shape, 7 + sum(shape), 3.0)
    if dtype == "bf16":
        x = S.to_bf16_rne(x)
    H, W, C, N = shape
    p, _ = gpu_quantize(to_dev(x, dtype, cuda_device), fmt, "grad", "hwcn", (N, C, H, W))
    assert_packed_equal(p, oracle.quantize(x, fmt, "grad", "hwcn"), f"hwcn {fmt} {dtype} {shape}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(16, 16, 3, 3), (32, 8, 1, 1), (8, 64, 5, 5)])
def test_oihw(cuda_device, fmt, shape):
    x = rand(shape, 3 + sum(shape), 0.05)
    p, _ = gpu_quantize(to_dev(x, "f32", cuda_device), fmt, "weight", "oihw", shape)
    assert_packed_equal(p, oracle.quantize(x, fmt, "weight", "oihw"), f"oihw {fmt} {shape}")


@pytest.mark.parametrize("fmt", FMTS)
def test_supplied_statistic(cuda_device, fmt):
    x = rand((16, 16, 4, 4), 99)
    for factor in (1.7, 0.3):
        amax_in = float(np.float32(np.abs(x).max() * factor))
        p, amax = gpu_quantize(to_dev(x, "f32", cuda_device), fmt, "act", "nchw", x.shape, amax_in=amax_in)
        ref = oracle.quantize(x, fmt, "act", "nchw", amax_in=amax_in)
        assert amax == ref["amax"]
        assert_packed_equal(p, ref, f"supplied statistic x{factor}")


@pytest.mark.parametrize("fmt", FMTS)
def test_rounding_midpoints(cuda_device, fmt):
    """Inputs exactly on, and one ulp either side of, every rounding midpoint."""
    from test_oracle_quantizer import midpoint_tensor
    x = midpoint_tensor(fmt)
    p, _ = gpu_quantize(to_dev(x, "f32", cuda_device), fmt, "act", "nchw", x.shape)
    assert_packed_equal(p, oracle.quantize(x, fmt, "act", "nchw"), "midpoints")


@pytest.mark.parametrize("fmt", FMTS)
def test_lossless_round_trip_values(cuda_device, fmt):
    """Quotients landing exactly on grid points and scale midpoints (a dense
    sweep of values k * 2^-j with few significant bits)."""
    rng = np.random.default_rng(5)
    x = (rng.integers(-64, 65, (16, 16, 4, 4)) * 2.0 ** -5).astype(np.float32)
    x[0, 0, 0, 0] = 448.0
    p, _ = gpu_quantize(to_dev(x, "f32", cuda_device), fmt, "act", "nchw", x.shape)
    assert_packed_equal(p, oracle.quantize(x, fmt, "act", "nchw"), "grid values")


def test_zero_tensor(cuda_device):
    x = np.zeros((8, 8, 2, 2), dtype=np.float32)
    x[:4] = -0.0
    p, amax = gpu_quantize(to_dev(x, "f32", cuda_device), "e2m1", "act", "nchw", x.shape)
    assert amax == 0.0
    assert_packed_equal(p, oracle.quantize(x, "e2m1", "act", "nchw"), "zeros")


def test_nonfinite_sets_status(cuda_device):
    import microscaling_quantized_convolution_only_b300 as mq
    x = np.ones((8, 8, 2, 2), dtype=np.float32)
    x[1, 2, 1, 0] = np.nan
    xd = to_dev(x, "f32", cuda_device)
    p = mq.Packed("e2m1", "act", x.shape, device=cuda_device)
    amax = torch.zeros(1, device=cuda_device)
    mq.quantize_cbf(xd, "nchw", p, amax_out=amax)
    st = mq.device_status()
    assert st & (1 << 4)
    assert mq.device_status() == 0    # cleared by the read


@pytest.mark.parametrize("wl_layer", [(2, 0), (3, 0), (4, 0), (5, 0)], ids=["r18-56", "yolo-320", "stack-fp4", "stack-fp6"])
def test_full_size_activation(cuda_device, wl_layer):
    """The largest activation tensor of each big workload, compared in full."""
    wl = S.WORKLOADS[wl_layer[0]]
    L = wl.layers[wl_layer[1]]
    x = S.draw_x(wl, wl_layer[1])
    p, amax = gpu_quantize(to_dev(x, wl.dtype, cuda_device), wl.fmt, "act", "nchw", L.x_shape())
    ref = oracle.quantize(x, wl.fmt, "act", "nchw")
    assert amax == ref["amax"]
    assert_packed_equal(p, ref, f"{wl.name} X")


def _tiny(shape, seed, amax):
    """A tensor scaled so that its amax is `amax` (fp32, subnormal values
    included when amax is small enough), with exact zeros, negative zeros and
    a few of the smallest subnormals mixed in."""
    x = np.random.default_rng(seed).standard_normal(shape)
    x = (x / np.abs(x).max() * amax).astype(np.float32)
    x.ravel()[::11] = 0.0
    x.ravel()[3::13] = -0.0
    x.ravel()[5::17] = np.float32(1.4e-45)            # 2^-149
    x.ravel()[7::19] = -np.float32(2.8e-45)
    x.ravel()[0] = np.float32(amax)
    return x


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("amax", [1e-20, 1e-36, 1e-40], ids=["Tscale-below-2^-62", "Tscale-subnormal",
                                                              "Tscale-deep-subnormal"])
@pytest.mark.parametrize("layout", ["nchw", "hwcn"])
def test_tiny_tensor_scale(cuda_device, fmt, amax, layout):
    """T_scale below 2^-62 and subnormal T_scale (amax ~1e-36, 1e-40), with
    subnormal inputs: codes and scales still bit-exact against the oracle."""
    shape = (16, 24, 6, 8)
    x = _tiny(shape, 11, amax)
    if layout == "hwcn":
        xs = np.ascontiguousarray(x.transpose(2, 3, 1, 0))
        p, a = gpu_quantize(to_dev(xs, "f32", cuda_device), fmt, "grad", layout, shape)
        ref = oracle.quantize(xs, fmt, "grad", layout)
    else:
        p, a = gpu_quantize(to_dev(x, "f32", cuda_device), fmt, "act", layout, shape)
        ref = oracle.quantize(x, fmt, "act", layout)
    assert a == ref["amax"]
    assert_packed_equal(p, ref, f"tiny T_scale amax={amax} {fmt} {layout}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("data_amax,stat", [(1.0, 1e-36), (1e20, 1e-30), (1e-30, 1e-38), (3e38, 1e-20)],
                         ids=["unit-data-subnormal-stat", "huge-data-tiny-stat", "tiny-data-subnormal-stat",
                              "max-data-tiny-stat"])
def test_supplied_statistic_far_below_data(cuda_device, fmt, data_amax, stat):
    """A supplied statistic far below the data: T_scale tiny or subnormal,
    most quotients saturate (some beyond 2^64 x T_scale); bit-exact against
    the oracle for both the bf16-pair and the fp32 code paths."""
    for dtype in ("f32", "bf16"):
        x = _tiny((16, 16, 4, 8), 21, data_amax)
        if dtype == "bf16":
            x = S.to_bf16_rne(x)
        p, _ = gpu_quantize(to_dev(x, dtype, cuda_device), fmt, "act", "nchw", x.shape, amax_in=stat)
        ref = oracle.quantize(x, fmt, "act", "nchw", amax_in=stat)
        assert_packed_equal(p, ref, f"data {data_amax} statistic {stat} {fmt} {dtype}")


EMAXV = {"e2m1": 6.0, "e2m3": 7.5, "e4m3": 448.0}


def tie_dense(shape, seed, fmt, exact):
    """ReLU(N(0,1)) in bf16 whose amax puts many quotients on or next to a
    rounding midpoint.  exact: amax = maxB_ef * 448 / 256, so T_scale = 2^-8
    exactly and quotients of few-bit bf16 values land exactly on midpoints.
    Otherwise amax = 5.46875 = 175/32, which shares factors with maxB_ef * 448
    (2688 = 2^7 * 21, 3360 = 2^5 * 105, 200704 = 2^12 * 49): T_scale is a
    short fraction rounded once to fp32, and quotients land within about
    2^-24 of midpoints, inside the 2^-20 bracket, yet not on them."""
    x = np.maximum(np.random.default_rng(seed).standard_normal(shape), 0).astype(np.float32)
    top = np.float32(EMAXV[fmt] * 448 / 256) if exact else np.float32(5.46875)
    x = S.to_bf16_rne(np.minimum(x * (top / np.float32(5.5) if exact else 1.0), top * 0.99).astype(np.float32))
    x.ravel()[0] = top
    return x


def near_midpoint_blocks(x, fmt, role, layout, stat=None):
    """Fraction of blocks whose oracle codes change when every input moves by
    a relative 2^-20 either way (same statistic, by default the amax): blocks
    with a quotient on or next to a rounding midpoint."""
    a = float(np.abs(x).max()) if stat is None else stat
    ends = [oracle.quantize((x.astype(np.float64) * (1 + d * 2.0 ** -20)).astype(np.float32), fmt, role, layout,
                            amax_in=a) for d in (-1, 1)]
    c0, c1 = (e["codes"].reshape(len(e["scales"]), -1) for e in ends)
    return float((c0 != c1).any(axis=1).mean())


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("exact", [False, True], ids=["near-ties", "exact-ties"])
@pytest.mark.parametrize("path", ["nchw-bf16-tma", "nchw-bf16-direct", "nchw-f32-tma", "hwcn-bf16"])
def test_tie_dense_inputs(cuda_device, fmt, exact, path):
    """Inputs with many quotients on, or within fp32 rounding of, a rounding
    midpoint (5 % to 70 % of blocks): every encoder path settles them exactly
    like the oracle, codes and scales bit for bit."""
    layout, dtype, shape = {"nchw-bf16-tma": ("nchw", "bf16", (32, 64, 16, 16)),
                            "nchw-bf16-direct": ("nchw", "bf16", (32, 64, 7, 7)),
                            "nchw-f32-tma": ("nchw", "f32", (32, 16, 8, 8)),
                            "hwcn-bf16": ("hwcn", "bf16", (6, 7, 64, 32))}[path]
    x = tie_dense(shape, 3, fmt, exact)
    role = "act" if layout == "nchw" else "grad"
    dims = shape if layout == "nchw" else (shape[3], shape[2], shape[0], shape[1])
    assert near_midpoint_blocks(x, fmt, role, layout) > 0.03
    p, a = gpu_quantize(to_dev(x, dtype, cuda_device), fmt, role, layout, dims)
    ref = oracle.quantize(x, fmt, role, layout)
    assert a == ref["amax"]
    assert_packed_equal(p, ref, f"tie-dense {path} {fmt} {'exact' if exact else 'near'}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("path", ["nchw-bf16-tma", "nchw-bf16-direct", "hwcn-f32"])
def test_codes_buffer_16_byte_aligned_only(cuda_device, fmt, path):
    """A codes buffer that starts 16 bytes past a 32-byte boundary (the
    alignment the ABI requires): every block payload then takes the 16-byte
    store path instead of the 32-byte one; codes and scales still bit-exact,
    and the bytes around the buffer untouched."""
    layout, dtype, shape = {"nchw-bf16-tma": ("nchw", "bf16", (16, 32, 8, 8)),
                            "nchw-bf16-direct": ("nchw", "bf16", (16, 32, 7, 5)),
                            "hwcn-f32": ("hwcn", "f32", (5, 6, 32, 16))}[path]
    x = rand(shape, 31)
    if dtype == "bf16":
        x = S.to_bf16_rne(x)
    role = "act" if layout == "nchw" else "grad"
    dims = shape if layout == "nchw" else (shape[3], shape[2], shape[0], shape[1])
    import microscaling_quantized_convolution_only_b300 as mq
    nc = mq.packed_code_bytes(fmt, dims)
    backing = torch.full((nc + 64,), 0xA5, dtype=torch.uint8, device=cuda_device)
    assert backing.data_ptr() % 32 == 0
    codes = backing[16:16 + nc]
    p = mq.Packed(fmt, role, dims, device=cuda_device, codes=codes)
    amax = torch.zeros(1, device=cuda_device)
    mq.quantize_cbf(to_dev(x, dtype, cuda_device), layout, p, amax_out=amax)
    mq.check_device_status()
    assert_packed_equal(p, oracle.quantize(x, fmt, role, layout), f"16-byte-aligned codes {path} {fmt}")
    rest = torch.cat([backing[:16], backing[16 + nc:]]).cpu()
    assert bool((rest == 0xA5).all()), "bytes outside the codes buffer were written"
