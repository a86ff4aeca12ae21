"""GPU parity of mqconv_fwd / mqconv_dgrad / mqconv_wgrad against the fp64
7-loop oracle on the same packed operands (MicroQonv §IV-A GEMMs).

Per element |gpu - oracle| <= 1e-5 * sum|a*b| + 1e-7, and relative L2 <= 1e-5.
Small layers are compared in full; the workloads' full-size layers on sampled
outputs computed one by one by the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic as S
from mqtest import LayerRun, check_close, hwcn_to_nchw
from synthetic import Layer

pytestmark = pytest.mark.gpu

SMALL = [
    Layer(8, 16, 8, 8, 16, 3, 1, 1),      # workload 0
    Layer(8, 16, 9, 7, 32, 3, 2, 1),      # stride 2, ragged
    Layer(16, 32, 6, 5, 24, 3, 1, 0),     # no padding
    Layer(8, 24, 10, 10, 16, 1, 2, 0),    # 1x1 stride 2
    Layer(8, 8, 5, 5, 8, 5, 1, 2),        # 5x5
    Layer(24, 48, 4, 6, 40, 3, 1, 1),     # ragged channels vs tile widths
    Layer(8, 16, 7, 7, 272, 3, 1, 1),     # more than 256 output channels
    Layer(8, 264, 3, 3, 16, 3, 2, 1),     # more than 256 input channels
    Layer(8, 16, 9, 8, 32, 3, 2, 1),      # stride 2, even width (halo column phases), ragged rows
    Layer(16, 32, 10, 14, 48, 3, 2, 1),   # stride 2, two channel chunks, ragged positions
    Layer(8, 32, 12, 12, 24, 1, 2, 0),    # 1x1 stride 2 through the halo path
    Layer(8, 16, 8, 6, 16, 3, 2, 0),      # stride 2 without padding
    Layer(24, 16, 14, 10, 136, 3, 2, 1),  # stride 2, three batch groups, two output-channel tiles
    Layer(8, 16, 11, 12, 16, 5, 2, 2),    # 5x5 stride 2 (three taps per column phase)
    Layer(8, 16, 8, 8, 16, 2, 2, 0),      # 2x2 stride 2 (one tap per output phase)
    Layer(16, 32, 9, 10, 16, 3, 2, 2),    # stride 2, padding 2 (dgrad phases start one row in)
]


def run_full(run: LayerRun, what):
    L = run.layer
    Xd, Wd, Gd = run.oracle_operands()
    Y, Ya = oracle.conv_fwd(Xd, Wd, L)
    check_close(hwcn_to_nchw(run.fwd()), Y, Ya, f"{what} fwd")
    dX, dXa = oracle.conv_dgrad(Wd, Gd, L)
    check_close(hwcn_to_nchw(run.dgrad()), dX, dXa, f"{what} dgrad")
    dW, dWa = oracle.conv_wgrad(Gd, Xd, L)
    check_close(run.wgrad().cpu().numpy(), dW, dWa, f"{what} wgrad")


@pytest.mark.parametrize("fmt", ["e2m1", "e2m3", "e4m3"])
@pytest.mark.parametrize("L", SMALL, ids=lambda L: L.name())
def test_small_layers_full(cuda_device, fmt, L):
    rng = np.random.default_rng(L.N + L.Cin + L.Cout)
    X = np.maximum(rng.standard_normal(L.x_shape()), 0).astype(np.float32)
    W = (rng.standard_normal(L.w_shape()) * np.sqrt(2 / (L.Cin * L.k * L.k))).astype(np.float32)
    dY = (rng.standard_normal(L.y_shape()) * 0.1).astype(np.float32)
    run_full(LayerRun(L, fmt, "f32", X, W, dY, cuda_device), f"{fmt} {L.name()}")


MIXED_LAYERS = [Layer(8, 16, 8, 8, 16, 3, 1, 1), Layer(16, 32, 10, 14, 48, 3, 2, 1), Layer(32, 64, 12, 12, 64, 3, 1, 1)]


@pytest.mark.parametrize("fmts", [("e2m1", "e4m3", "e2m3"), ("e4m3", "e2m1", "e4m3"), ("e2m3", "e2m3", "e2m1")],
                         ids=lambda f: "-".join(f))
@pytest.mark.parametrize("L", MIXED_LAYERS, ids=lambda L: L.name())
def test_mixed_formats(cuda_device, fmts, L):
    """MicroQonv+: X, W and dY each in their own element format; every GEMM
    mixes two formats (fp16 decode of each operand, E4M3 pairs pre-scaled)."""
    rng = np.random.default_rng(L.N + 3 * L.Cin + L.Cout)
    X = np.maximum(rng.standard_normal(L.x_shape()), 0).astype(np.float32)
    W = (rng.standard_normal(L.w_shape()) * np.sqrt(2 / (L.Cin * L.k * L.k))).astype(np.float32)
    dY = (rng.standard_normal(L.y_shape()) * 0.1).astype(np.float32)
    run_full(LayerRun(L, fmts, "f32", X, W, dY, cuda_device), f"{fmts} {L.name()}")


@pytest.mark.parametrize("li", range(5))
def test_workload1_full(cuda_device, li):
    wl = S.WORKLOADS[1]
    L = wl.layers[li]
    run = LayerRun(L, wl.fmt, wl.dtype, S.draw_x(wl, li), S.draw_w(wl, li), S.draw_dy(wl, li), cuda_device)
    run_full(run, f"resnet32 layer {li}")


def test_workload0_full(cuda_device):
    wl = S.WORKLOADS[0]
    L = wl.layers[0]
    run_full(LayerRun(L, wl.fmt, wl.dtype, S.draw_x(wl, 0), S.draw_w(wl, 0), S.draw_dy(wl, 0), cuda_device),
             "tiny")


def sample_indices(shape, count, seed):
    """Random flat indices plus every border position of a few (n, c) planes."""
    rng = np.random.default_rng(seed)
    total = int(np.prod(shape))
    idx = rng.integers(0, total, count)
    n_, c_, h_, w_ = shape
    border = []
    for n, c in ((0, 0), (n_ - 1, c_ - 1), (n_ // 2, c_ // 3)):
        for h in range(h_):
            for w in range(w_):
                if h in (0, h_ - 1) or w in (0, w_ - 1):
                    border.append(((n * c_ + c) * h_ + h) * w_ + w)
    return np.unique(np.concatenate([idx, np.asarray(border, dtype=np.int64)]))


def run_sampled(run: LayerRun, what, n_fwd=4096, n_wg=128):
    L = run.layer
    Xd, Wd, Gd = run.oracle_operands()
    y = hwcn_to_nchw(run.fwd()).ravel()
    idx = sample_indices(L.y_shape(), n_fwd, 1)
    ref, refa = oracle.conv_fwd_at(Xd, Wd, L, idx)
    check_close(y[idx], ref, refa, f"{what} fwd (sampled)")
    dx = hwcn_to_nchw(run.dgrad()).ravel()
    idx = sample_indices(L.x_shape(), n_fwd, 2)
    ref, refa = oracle.conv_dgrad_at(Wd, Gd, L, idx)
    check_close(dx[idx], ref, refa, f"{what} dgrad (sampled)")
    dw = run.wgrad().cpu().numpy().ravel()
    rng = np.random.default_rng(3)
    idx = np.unique(np.concatenate([rng.integers(0, dw.size, n_wg), [0, dw.size - 1]]))
    ref, refa = oracle.conv_wgrad_at(Gd, Xd, L, idx)
    check_close(dw[idx], ref, refa, f"{what} wgrad (sampled)")


@pytest.mark.parametrize("wi,li", [(2, i) for i in range(10)] + [(3, i) for i in range(8)],
                         ids=lambda v: str(v))
def test_workload_layers_sampled(cuda_device, wi, li):
    wl = S.WORKLOADS[wi]
    L = wl.layers[li]
    run = LayerRun(L, wl.fmt, wl.dtype, S.draw_x(wl, li), S.draw_w(wl, li), S.draw_dy(wl, li), cuda_device,
                   check_quant=(li < 2))
    run_sampled(run, f"{wl.name} layer {li}", n_wg=64)
