"""GPU test of mqconv_wgrad_noalloc, the weight-gradient entry point that
allocates no device memory, for callers that cannot give the library extra
memory (a fixed device-memory budget owned by the host runtime, an allocator
that must not be bypassed, or code that cannot afford the synchronisation an
allocation may cause).

Each case calls it twice in a row and checks both results against the
oracle's dW (MicroQonv §IV-A: G_W = G_Y X'^T) and against mqconv_wgrad, the
entry point that takes a workspace, with the tolerance the conv parity tests
use, |a - b| <= 1e-5 sum|a*b| + 1e-7 per element and relative L2 <= 1e-5.
The two entry points may differ only in the order the split-K partial sums
are added.  This file is collected last so that a run stopping at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import microscaling_quantized_convolution_only_b300 as mq
import oracle
import synthetic as S
from mqtest import LayerRun, check_close
from synthetic import Layer

pytestmark = pytest.mark.gpu

CASES = [
    (S.WORKLOADS[0], S.WORKLOADS[0].layers[0], "tiny layer"),
    # large reduction: the built-in scratch forces fewer, longer split-K chunks
    (S.WORKLOADS[2], S.scaled_layer(S.WORKLOADS[2].layers[1], N=32), "28x28 C128 layer, N=32"),
    # stride 2 with an odd width runs on the generic kernel; its plan wants 45
    # splits of 589,824 bytes, the scratch holds 28, so the cap re-splits it
    (S.WORKLOADS[2], Layer(64, 128, 29, 29, 128, 3, 2, 1), "29x29 C128 stride-2 layer, generic kernel"),
]


@pytest.mark.parametrize("wl,L,name", CASES, ids=[c[2] for c in CASES])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(cuda_device, wl, L, name):
    X = S.draw_x(wl, 0, L.x_shape())
    W = S.draw_w(wl, 0, L.w_shape())
    dY = S.draw_dy(wl, 0, L.y_shape())
    run = LayerRun(L, wl.fmt, wl.dtype, X, W, dY, cuda_device, check_quant=False)
    Xd, _, Gd = run.oracle_operands()
    ref, refa = oracle.conv_wgrad(Gd, Xd, L)
    with_ws = run.wgrad().cpu().numpy().astype(np.float64)
    check_close(with_ws, ref, refa, f"{name}, workspace entry point vs oracle")
    for call in range(2):
        dw = torch.full(L.w_shape(), float("nan"), device=cuda_device)
        mq.wgrad_noalloc(L, run.gq, run.xq, dw)
        mq.check_device_status()
        got = dw.cpu().numpy()
        check_close(got, ref, refa, f"{name}, no-alloc call {call + 1} vs oracle")
        check_close(got, with_ws, refa, f"{name}, no-alloc call {call + 1} vs workspace entry point")


def test_noalloc_rejects_partial_sums_beyond_scratch(cuda_device):
    # Cout * Kh * Kw * Cin fp32 = 1024 * 9 * 512 * 4 bytes > the built-in scratch
    L = Layer(8, 512, 1, 1, 1024, 3, 1, 1)
    xq = mq.Packed("e2m1", "act", L.x_shape(), device=cuda_device)
    gq = mq.Packed("e2m1", "grad", L.y_shape(), device=cuda_device)
    dw = torch.empty(L.w_shape(), device=cuda_device)
    with pytest.raises(mq.MQError, match="workspace"):
        mq.wgrad_noalloc(L, gq, xq, dw)
