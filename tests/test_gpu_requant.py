"""GPU parity of the fused requantizing epilogues (mqconv_fwd with mq_requant,
mqconv_dgrad_requant): the output goes from the accumulators straight into
packed 8x8 CBF blocks, its T_scale built from a caller-supplied statistic
(the Hindsight scheme of MicroQonv §VII).

The reference is the oracle quantizer applied, with the same statistic, to the
fp32 result the same kernels write without the epilogue (identical mainloop
and accumulation order, so identical fp32 values): codes, scales and T_scale
must match bit for bit, and amax_out must equal max |result|.  The fp32
output written alongside the packed one must equal the unfused output.
"""
import numpy as np
import pytest
import torch

import microscaling_quantized_convolution_only_b300 as mq
import oracle
import synthetic as S
from mqtest import LayerRun, assert_packed_equal, check_close, hwcn_to_nchw
from synthetic import Layer

pytestmark = pytest.mark.gpu

LAYERS = [
    Layer(8, 16, 8, 8, 16, 3, 1, 1),      # halo kernel, tiny
    Layer(16, 32, 9, 7, 48, 3, 1, 1),     # halo kernel, ragged positions
    Layer(8, 16, 9, 7, 32, 3, 2, 1),      # generic kernel (stride 2)
    Layer(8, 24, 10, 10, 16, 1, 2, 0),    # generic kernel (1x1 stride 2)
    Layer(32, 64, 12, 12, 64, 3, 1, 1),   # halo kernel, several tiles
    Layer(16, 32, 10, 14, 48, 3, 2, 1),   # halo kernel, stride 2
]


def _inputs(L, seed):
    rng = np.random.default_rng(seed)
    X = np.maximum(rng.standard_normal(L.x_shape()), 0).astype(np.float32)
    W = (rng.standard_normal(L.w_shape()) * np.sqrt(2 / (L.Cin * L.k * L.k))).astype(np.float32)
    dY = (rng.standard_normal(L.y_shape()) * 0.1).astype(np.float32)
    return X, W, dY


def _check(packed, ref_hwcn, fmt, role, stat, amax_out, what):
    ref = oracle.quantize(ref_hwcn, fmt, role, "hwcn", amax_in=stat)
    assert_packed_equal(packed, ref, what)
    assert float(amax_out.item()) == float(np.max(np.abs(ref_hwcn))), f"{what}: amax_out"


@pytest.mark.parametrize("fmt_in,fmt_out", [("e2m1", "e2m1"), ("e2m3", "e2m3"), ("e4m3", "e4m3"), ("e2m1", "e2m3")])
@pytest.mark.parametrize("L", LAYERS, ids=lambda L: L.name())
@pytest.mark.parametrize("factor", [1.0, 1.7])
def test_fwd_requant(cuda_device, fmt_in, fmt_out, L, factor):
    run = LayerRun(L, fmt_in, "f32", *_inputs(L, L.N + L.Cout), cuda_device, check_quant=False)
    y = run.fwd()
    y_np = y.cpu().numpy()
    stat = float(np.float32(np.max(np.abs(y_np)) * factor))
    out = mq.Packed(fmt_out, "act", L.y_shape(), device=cuda_device)
    ain = torch.tensor([stat], device=cuda_device)
    aout = torch.zeros(1, device=cuda_device)
    y2 = torch.full_like(y, float("nan"))
    mq.fwd(L, run.xq, run.wq, y2, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
    mq.check_device_status()
    assert torch.equal(y2, y), "fp32 output beside the fused epilogue differs from the unfused one"
    _check(out, y_np, fmt_out, "act", stat, aout, f"fwd requant {fmt_in}->{fmt_out} {L.name()}")
    # packed output only
    out2 = mq.Packed(fmt_out, "act", L.y_shape(), device=cuda_device)
    mq.fwd(L, run.xq, run.wq, None, rq_out=out2, rq_amax_in=ain, rq_amax_out=aout)
    mq.check_device_status()
    assert torch.equal(out2.codes, out.codes) and torch.equal(out2.scales, out.scales)


@pytest.mark.parametrize("fmt_in,fmt_out", [("e2m1", "e2m1"), ("e2m3", "e2m3"), ("e4m3", "e4m3")])
@pytest.mark.parametrize("L", LAYERS, ids=lambda L: L.name())
def test_dgrad_requant(cuda_device, fmt_in, fmt_out, L):
    run = LayerRun(L, fmt_in, "f32", *_inputs(L, 7 + L.N), cuda_device, check_quant=False)
    dx = run.dgrad()
    dx_np = dx.cpu().numpy()
    stat = float(np.float32(np.max(np.abs(dx_np)) * 1.25))
    out = mq.Packed(fmt_out, "grad", L.x_shape(), device=cuda_device)
    ain = torch.tensor([stat], device=cuda_device)
    aout = torch.zeros(1, device=cuda_device)
    dx2 = torch.full_like(dx, float("nan"))
    mq.dgrad(L, run.wq, run.gq, dx2, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
    mq.check_device_status()
    assert torch.equal(dx2, dx), "fp32 dX beside the fused epilogue differs from the unfused one"
    _check(out, dx_np, fmt_out, "grad", stat, aout, f"dgrad requant {fmt_in}->{fmt_out} {L.name()}")
    out2 = mq.Packed(fmt_out, "grad", L.x_shape(), device=cuda_device)
    mq.dgrad(L, run.wq, run.gq, None, rq_out=out2, rq_amax_in=ain, rq_amax_out=aout)
    mq.check_device_status()
    assert torch.equal(out2.codes, out.codes) and torch.equal(out2.scales, out.scales)


def test_stack_layer_requant_full_size(cuda_device):
    """The 56x56 C128 stack layer (batch 64) in NVFP4: fused fwd and dgrad
    epilogues against the oracle quantizer on the unfused fp32 results."""
    wl = S.WORKLOADS[4]
    L = S.scaled_layer(wl.layers[0], N=64)
    X = S.draw_x(wl, 0, L.x_shape())
    W = S.draw_w(wl, 0, L.w_shape())
    dY = S.draw_dy(wl, 0, L.y_shape())
    run = LayerRun(L, wl.fmt, wl.dtype, X, W, dY, cuda_device, check_quant=False)
    for op, role, shape in (("fwd", "act", L.y_shape()), ("dgrad", "grad", L.x_shape())):
        ref = run.fwd() if op == "fwd" else run.dgrad()
        ref_np = ref.cpu().numpy()
        stat = float(np.float32(np.max(np.abs(ref_np))))
        out = mq.Packed(wl.fmt, role, shape, device=cuda_device)
        ain = torch.tensor([stat], device=cuda_device)
        aout = torch.zeros(1, device=cuda_device)
        if op == "fwd":
            mq.fwd(L, run.xq, run.wq, None, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
        else:
            mq.dgrad(L, run.wq, run.gq, None, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
        mq.check_device_status()
        _check(out, ref_np, wl.fmt, role, stat, aout, f"stack layer {op} requant")


def test_requant_rejects_wrong_role(cuda_device):
    L = LAYERS[0]
    run = LayerRun(L, "e2m1", "f32", *_inputs(L, 3), cuda_device, check_quant=False)
    out = mq.Packed("e2m1", "act", L.x_shape(), device=cuda_device)     # dgrad wants role grad
    ain = torch.ones(1, device=cuda_device)
    with pytest.raises(mq.MQError, match="invalid argument"):
        mq.dgrad(L, run.wq, run.gq, None, rq_out=out, rq_amax_in=ain)


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
@pytest.mark.parametrize("L", [LAYERS[0], LAYERS[2]], ids=["halo", "generic"])
@pytest.mark.parametrize("stat_factor", [1.0, 1e-16], ids=["Tscale-below-2^-62", "Tscale-subnormal"])
def test_requant_tiny_tensor_scale(cuda_device, fmt, L, stat_factor):
    """Activations scaled by 1e-20: Y ~ 1e-20, so its T_scale (from a
    statistic of max|Y|, or that times 1e-16 -- subnormal) is below 2^-62 and
    the fused epilogues encode through their tiny-scale path.  Bit-exact
    against the oracle quantizer on the unfused fp32 output."""
    X, W, dY = _inputs(L, 5 + L.N)
    run = LayerRun(L, fmt, "f32", (X * np.float32(1e-20)).astype(np.float32), W,
                   (dY * np.float32(1e-20)).astype(np.float32), cuda_device, check_quant=True)
    for op, role, shape in (("fwd", "act", L.y_shape()), ("dgrad", "grad", L.x_shape())):
        ref = run.fwd() if op == "fwd" else run.dgrad()
        ref_np = ref.cpu().numpy()
        stat = float(np.float32(np.max(np.abs(ref_np)) * stat_factor))
        assert 0.0 < stat < 1e-18
        out = mq.Packed(fmt, role, shape, device=cuda_device)
        ain = torch.tensor([stat], device=cuda_device)
        aout = torch.zeros(1, device=cuda_device)
        if op == "fwd":
            mq.fwd(L, run.xq, run.wq, None, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
        else:
            mq.dgrad(L, run.wq, run.gq, None, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
        mq.check_device_status()
        _check(out, ref_np, fmt, role, stat, aout, f"{op} requant tiny T_scale x{stat_factor} {fmt} {L.name()}")


CHANNEL_LAYERS = [
    Layer(16, 128, 9, 7, 128, 3, 1, 1),    # 128 channels both ways, ragged positions
    Layer(8, 128, 6, 10, 256, 3, 1, 1),    # two output-channel tiles forward, one batch group
    Layer(32, 256, 5, 5, 128, 1, 1, 0),    # 1x1, four batch groups, more input channels than a tile
]


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
@pytest.mark.parametrize("L", CHANNEL_LAYERS, ids=lambda L: L.name())
@pytest.mark.parametrize("scale", [1.0, 1e-20], ids=["unit", "tiny-Tscale"])
def test_requant_many_channels(cuda_device, fmt, L, scale):
    """Stride-1 layers with 128 or more channels (several output-channel
    tiles, several input-channel chunks): fp32 outputs against the oracle, and
    the fused requantizations bit-exact against the oracle quantizer on the
    unfused fp32 outputs, at unit scale and with T_scale below 2^-62."""
    X, W, dY = _inputs(L, 11 + L.N)
    run = LayerRun(L, fmt, "f32", (X * np.float32(scale)).astype(np.float32), W,
                   (dY * np.float32(scale)).astype(np.float32), cuda_device, check_quant=True)
    Xd, Wd, Gd = run.oracle_operands()
    for op, role, shape in (("fwd", "act", L.y_shape()), ("dgrad", "grad", L.x_shape())):
        ref = run.fwd() if op == "fwd" else run.dgrad()
        want, wanta = oracle.conv_fwd(Xd, Wd, L) if op == "fwd" else oracle.conv_dgrad(Wd, Gd, L)
        check_close(hwcn_to_nchw(ref), want, wanta, f"{op} {fmt} {L.name()} x{scale}")
        ref_np = ref.cpu().numpy()
        stat = float(np.float32(np.max(np.abs(ref_np)) * 1.3))
        out = mq.Packed(fmt, role, shape, device=cuda_device)
        ain = torch.tensor([stat], device=cuda_device)
        aout = torch.zeros(1, device=cuda_device)
        y2 = torch.full_like(ref, float("nan"))
        if op == "fwd":
            mq.fwd(L, run.xq, run.wq, y2, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
        else:
            mq.dgrad(L, run.wq, run.gq, y2, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
        mq.check_device_status()
        assert torch.equal(y2, ref), f"{op}: fp32 output beside the fused epilogue differs from the unfused one"
        _check(out, ref_np, fmt, role, stat, aout, f"{op} requant {fmt} {L.name()} x{scale}")


EMAXV = {"e2m1": 6.0, "e2m3": 7.5, "e4m3": 448.0}


def _single_product_inputs(L, fmt, seed):
    """Sparse operands under which every output of fwd and dgrad is a single
    product of two dequantized values (or zero): X nonzero only in channel 0,
    dY only in channel 0, both only at rows and columns that are multiples of
    4 (any three consecutive rows or columns hold at most one).  The amax of X,
    W and dY are maxB_ef * 448 times powers of two, so their T_scale are exact
    powers of two and each product has few significant bits: its quotients
    land on, or next to, rounding midpoints of the requantized grid."""
    rng = np.random.default_rng(seed)
    e = np.float32(EMAXV[fmt] * 448)
    X = np.zeros(L.x_shape(), np.float32)
    X[:, 0, ::4, ::4] = np.maximum(rng.standard_normal(X[:, 0, ::4, ::4].shape), 0)
    X = (X / X.max() * e * np.float32(2.0 ** -8)).astype(np.float32)
    X[0, 0, 0, 0] = e * np.float32(2.0 ** -8)
    W = rng.standard_normal(L.w_shape()).astype(np.float32)
    W = (W / np.abs(W).max() * e * np.float32(0.9 * 2.0 ** -10)).astype(np.float32)
    W[0, 0, 0, 0] = e * np.float32(2.0 ** -10)
    dY = np.zeros(L.y_shape(), np.float32)
    dY[:, 0, ::4, ::4] = rng.standard_normal(dY[:, 0, ::4, ::4].shape)
    dY = (dY / np.abs(dY).max() * e * np.float32(0.9 * 2.0 ** -6)).astype(np.float32)
    dY[0, 0, 0, 0] = e * np.float32(2.0 ** -6)
    return X, W, dY


def _tie_stat(amax, fmt, exact):
    """maxB_ef * 448 times the power of two nearest amax / (maxB_ef * 448)
    (T_scale exact: quotients exactly on midpoints), else 175/32 times a
    power of two (T_scale a short fraction rounded once: quotients within
    fp32 rounding of midpoints)."""
    base = EMAXV[fmt] * 448 if exact else 5.46875
    return float(np.float32(base * 2.0 ** round(np.log2(amax / base))))


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
@pytest.mark.parametrize("L", [LAYERS[1], LAYERS[3], LAYERS[5]], ids=["halo", "generic-1x1-s2", "halo-s2"])
def test_requant_tie_dense(cuda_device, fmt, L):
    """Fused fwd and dgrad epilogues on outputs whose quotients sit on, or
    within fp32 rounding of, rounding midpoints: bit-exact against the oracle
    quantizer on the unfused fp32 results with the same statistic."""
    from test_gpu_quantize import near_midpoint_blocks
    run = LayerRun(L, fmt, "f32", *_single_product_inputs(L, fmt, L.N + L.Cin), cuda_device, check_quant=True)
    assert float(run.xq.s_t.item()) == 2.0 ** -8 and float(run.wq.s_t.item()) == 2.0 ** -10
    for op, role, shape in (("fwd", "act", L.y_shape()), ("dgrad", "grad", L.x_shape())):
        ref_np = (run.fwd() if op == "fwd" else run.dgrad()).cpu().numpy()
        for exact in (True, False):
            stat = _tie_stat(float(np.max(np.abs(ref_np))), fmt, exact)
            if exact:
                assert near_midpoint_blocks(ref_np, fmt, role, "hwcn", stat) > 0.005
            out = mq.Packed(fmt, role, shape, device=cuda_device)
            ain = torch.tensor([stat], device=cuda_device)
            aout = torch.zeros(1, device=cuda_device)
            if op == "fwd":
                mq.fwd(L, run.xq, run.wq, None, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
            else:
                mq.dgrad(L, run.wq, run.gq, None, rq_out=out, rq_amax_in=ain, rq_amax_out=aout)
            mq.check_device_status()
            _check(out, ref_np, fmt, role, stat, aout, f"tie-dense {op} requant {fmt} {L.name()} exact={exact}")
