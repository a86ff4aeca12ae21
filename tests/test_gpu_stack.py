"""Parity of the benchmarked configuration: the chained 4-layer stack
(N=256, 56x56, C 128->128, 3x3, stride 1, pad 1, bf16 inputs) in NVFP4 and
in the 6-bit variant, run through bench.py's own StackStep -- the exact
launches, tile plans (including the 49-way split-K weight gradient over
K = 802,816) and fused epilogues that the benchmark times.

After a first step (which sets the previous-step statistics of the fused
epilogues, the Hindsight scheme of MicroQonv §VII), one more step runs and
is checked in full against the oracle:

  * X0, W0..W3 and dY3 quantized once: codes, scales, T_scale bit-exact
    (MicroQonv §III-A, §IV-B);
  * every layer's Y, dX and dW against the explicit-im2col fp64 GEMM form of
    the oracle (MicroQonv §II-C, §IV-A) on the whole tensor, per element
    |gpu - oracle| <= 1e-5 sum|a*b| + 1e-7 and relative L2 <= 1e-5, on the
    packed operands the step itself produced;
  * every fused requantization (Y_l -> X_{l+1}, dX_l -> dY_{l-1}) bit-exact
    against the oracle quantizer applied, with the statistic the step used,
    to the fp32 result of the same kernel without the epilogue (identical
    accumulation order), and its amax output equal to max |result|.
"""
import numpy as np
import pytest
import torch

import bench
import microscaling_quantized_convolution_only_b300 as mq
import oracle
import synthetic as S
from mqtest import assert_packed_equal, check_close, hwcn_to_nchw, packed_to_oracle

pytestmark = pytest.mark.gpu


def _deq(p):
    return oracle.dequantize(packed_to_oracle(p))


@pytest.mark.parametrize("wi", [4, 5], ids=["nvfp4", "e2m3"])
def test_benched_stack_step_matches_oracle(cuda_device, wi):
    wl = S.WORKLOADS[wi]
    step = bench.StackStep(wl, cuda_device)
    L, nl, fmt = step.L, step.nl, step.fmt
    assert L.N == 256 and nl == 4
    step.run()
    torch.cuda.synchronize()
    y_stat = step.y_stat.cpu().numpy().copy()      # the statistics the checked step uses
    dx_stat = step.dx_stat.cpu().numpy().copy()
    step.run()
    torch.cuda.synchronize()
    mq.check_device_status()
    report = []

    # ---- tensors quantized once from the step's dense inputs
    ref = oracle.quantize(step.h_x0.float().numpy(), fmt, "act", "nchw")
    assert_packed_equal(step.xq[0], ref, "X0")
    assert float(step.amax[0].item()) == ref["amax"]
    for l in range(nl):
        assert_packed_equal(step.wq[l], oracle.quantize(step.h_w[l].float().numpy(), fmt, "weight", "oihw"), f"W{l}")
    ref = oracle.quantize(step.h_dy.float().numpy(), fmt, "grad", "nchw")
    assert_packed_equal(step.gq[nl - 1], ref, "dY3")
    del ref

    for l in range(nl):
        Xd, Wd = _deq(step.xq[l]), _deq(step.wq[l])
        # forward
        if l < nl - 1:
            y = torch.empty_like(step.y_last)
            mq.fwd(L, step.xq[l], step.wq[l], y)
            mq.check_device_status()
        else:
            y = step.y_last
        yr, yra = oracle.conv_fwd_gemm(Xd, Wd, L)
        report.append(("fwd", l, check_close(hwcn_to_nchw(y), yr, yra, f"{wl.name} layer {l} fwd")))
        del yr, yra
        if l < nl - 1:   # Y_l requantized by the fused epilogue into X_{l+1}
            y_np = y.cpu().numpy()
            q = oracle.quantize(y_np, fmt, "act", "hwcn", amax_in=float(y_stat[l]))
            assert_packed_equal(step.xq[l + 1], q, f"layer {l} fused requant of Y into X{l + 1}")
            assert float(step.y_amax[l].item()) == float(np.max(np.abs(y_np)))
            del y_np, q
        del y
        # data gradient
        Gd = _deq(step.gq[l])
        if l > 0:
            dx = torch.empty_like(step.dx)
            mq.dgrad(L, step.wq[l], step.gq[l], dx)
            mq.check_device_status()
        else:
            dx = step.dx
        dr, dra = oracle.conv_dgrad_gemm(Wd, Gd, L)
        report.append(("dgrad", l, check_close(hwcn_to_nchw(dx), dr, dra, f"{wl.name} layer {l} dgrad")))
        del dr, dra
        if l > 0:        # dX_l requantized by the fused epilogue into dY_{l-1}
            dx_np = dx.cpu().numpy()
            q = oracle.quantize(dx_np, fmt, "grad", "hwcn", amax_in=float(dx_stat[l]))
            assert_packed_equal(step.gq[l - 1], q, f"layer {l} fused requant of dX into dY{l - 1}")
            assert float(step.dx_amax[l].item()) == float(np.max(np.abs(dx_np)))
            del dx_np, q
        del dx
        # weight gradient (split-K over N Ho Wo = 802,816)
        wr, wra = oracle.conv_wgrad_gemm(Gd, Xd, L)
        report.append(("wgrad", l, check_close(step.dw[l].cpu().numpy(), wr, wra, f"{wl.name} layer {l} wgrad")))
        del Xd, Wd, Gd, wr, wra
    for op, l, (worst, rel) in report:
        print(f"{wl.name} layer {l} {op}: worst err/bound {worst:.3g}, relative L2 {rel:.3g}")
