"""Failure detection on the GPU without a GPU fault.

Every wait inside the convolution kernels is bounded.  The test withholds one
plain barrier arrival (the barrier of CTA 0's first accumulator slot expects
one release more than its epilogue warps give: no copy and no MMA is waiting
on it), with the kernels' 2 s wait limit, and checks that

  * the call returns and the device status word reports MQ_ERR_TIMEOUT,
  * nothing else is reported and the status word is cleared by the read,
  * the next normal call on the same stream gives the same result as before
    the fault, and that result matches the oracle on sampled outputs.

Nothing traps, faults or hangs: the expiring wait raises the CTA's abort
flag, the other warps leave their loops, the copies and MMAs already issued
are drained, and the tensor memory is freed before the CTA exits."""
import time

import numpy as np
import pytest
import torch

import microscaling_quantized_convolution_only_b300 as mq
import oracle
from mqtest import LayerRun, check_close, hwcn_to_nchw
from synthetic import Layer

pytestmark = pytest.mark.gpu

TIMEOUT_BIT = 1 << 5


def _sampled_fwd_check(run, y, what):
    L = run.layer
    Xd, Wd, _ = run.oracle_operands()
    idx = np.random.default_rng(4).integers(0, int(np.prod(L.y_shape())), 512)
    ref, refa = oracle.conv_fwd_at(Xd, Wd, L, idx)
    check_close(hwcn_to_nchw(y).ravel()[idx], ref, refa, what)


def test_withheld_release_times_out_and_context_survives(cuda_device):
    # 392 tiles of the halo forward kernel on <= 148 CTAs: CTA 0 runs a second
    # tile, whose first accumulator waits for the withheld release
    L = Layer(64, 128, 56, 56, 128, 3, 1, 1)
    rng = np.random.default_rng(9)
    X = np.maximum(rng.standard_normal(L.x_shape()), 0).astype(np.float32)
    W = (rng.standard_normal(L.w_shape()) * np.sqrt(2 / (L.Cin * 9))).astype(np.float32)
    dY = np.zeros(L.y_shape(), dtype=np.float32)
    run = LayerRun(L, "e2m1", "f32", X, W, dY, cuda_device, check_quant=False)
    before = run.fwd()
    assert mq.device_status() == 0

    y = torch.full_like(before, float("nan"))
    mq.test_fault_inject("withhold_acc_release")     # the issuer's wait expires after 2 s
    try:
        t0 = time.monotonic()
        mq.fwd(L, run.xq, run.wq, y)
        status = mq.device_status()                               # synchronizes
        elapsed = time.monotonic() - t0
    finally:
        mq.test_fault_inject("none")
    assert status & TIMEOUT_BIT, f"status {status:#x}: the withheld release did not expire a wait"
    assert status == TIMEOUT_BIT, f"status {status:#x}: unexpected bits beside the timeout"
    assert elapsed < 20.0
    assert mq.device_status() == 0, "the status word is cleared by the read"

    after = run.fwd()          # raises if the status word reports anything
    assert torch.equal(after, before), "the call after the fault differs from the one before it"
    _sampled_fwd_check(run, after, "forward after the fault")

