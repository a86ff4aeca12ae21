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
