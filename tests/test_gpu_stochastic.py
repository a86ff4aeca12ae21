"""GPU parity of stochastic rounding (MicroQonv §III-A: Round is
round-to-nearest or stochastic; the paper rounds gradients stochastically).

mqconv_quantize_cbf_sr and the fused epilogues with MQ_ROUND_SR against the
oracle's stochastic quantizer with the same Philox seed: codes, scales and
T_scale bit for bit.  The oracle's own pins (known answers of the generator,
neighbouring grid values, unbiasedness over seeds) are in
test_oracle_stochastic.py."""
import numpy as np
import pytest
import torch

import microscaling_quantized_convolution_only_b300 as mq
import oracle
import synthetic as S
from mqtest import LayerRun, assert_packed_equal, to_dev

pytestmark = pytest.mark.gpu
FMTS = ["e2m1", "e2m3", "e4m3"]
SEED = 0x9E3779B97F4A7C15


def _q_sr(x_dev, fmt, role, layout, dims, seed, amax_in=None):
    p = mq.Packed(fmt, role, dims, device=x_dev.device)
    aout = torch.zeros(1, device=x_dev.device)
    ain = None if amax_in is None else torch.tensor([amax_in], dtype=torch.float32, device=x_dev.device)
    mq.quantize_cbf(x_dev, layout, p, amax_in=ain, amax_out=aout, sr_seed=seed)
    mq.check_device_status()
    return p


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(8, 16, 8, 8), (16, 24, 7, 5), (64, 32, 3, 9), (16, 136, 6, 12)])
def test_quantize_sr_nchw(cuda_device, fmt, dtype, shape):
    x = (np.random.default_rng(sum(shape)).standard_normal(shape) * 0.03).astype(np.float32)
    if dtype == "bf16":
        x = S.to_bf16_rne(x)
    x.ravel()[::7] = 0.0
    p = _q_sr(to_dev(x, dtype, cuda_device), fmt, "grad", "nchw", shape, SEED)
    assert_packed_equal(p, oracle.quantize(x, fmt, "grad", "nchw", sr_seed=SEED), f"SR nchw {fmt} {dtype} {shape}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_quantize_sr_hwcn_and_statistic(cuda_device, fmt, dtype):
    H, W, C, N = 5, 6, 24, 16
    x = (np.random.default_rng(5).standard_normal((H, W, C, N)) * 2.0).astype(np.float32)
    if dtype == "bf16":
        x = S.to_bf16_rne(x)
    for seed, stat in ((1, None), (2 ** 63 + 12345, float(np.abs(x).max()) * 1.3)):
        p = _q_sr(to_dev(x, dtype, cuda_device), fmt, "grad", "hwcn", (N, C, H, W), seed, amax_in=stat)
        assert_packed_equal(p, oracle.quantize(x, fmt, "grad", "hwcn", amax_in=stat, sr_seed=seed),
                            f"SR hwcn {fmt} {dtype} seed {seed}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("amax", [1e-20, 1e-38])
def test_quantize_sr_tiny_tensor_scale(cuda_device, fmt, amax):
    x = np.random.default_rng(6).standard_normal((16, 16, 4, 4))
    x = (x / np.abs(x).max() * amax).astype(np.float32)
    p = _q_sr(to_dev(x, "f32", cuda_device), fmt, "grad", "nchw", x.shape, 77)
    assert_packed_equal(p, oracle.quantize(x, fmt, "grad", "nchw", sr_seed=77), f"SR tiny {amax} {fmt}")


def test_quantize_sr_seed_changes_codes_and_is_deterministic(cuda_device):
    x = to_dev(np.random.default_rng(2).standard_normal((16, 32, 6, 6)).astype(np.float32), "f32", cuda_device)
    a = _q_sr(x, "e2m1", "grad", "nchw", (16, 32, 6, 6), 10)
    b = _q_sr(x, "e2m1", "grad", "nchw", (16, 32, 6, 6), 10)
    c = _q_sr(x, "e2m1", "grad", "nchw", (16, 32, 6, 6), 11)
    assert torch.equal(a.codes, b.codes) and not torch.equal(a.codes, c.codes)
    assert torch.equal(a.scales, c.scales)


LAYERS = [
    S.Layer(16, 32, 9, 7, 48, 3, 1, 1),     # halo kernel
    S.Layer(8, 16, 9, 7, 32, 3, 2, 1),      # generic kernel (odd width at stride 2)
    S.Layer(16, 32, 10, 14, 48, 3, 2, 1),   # halo kernel, stride-2 data gradient as output quads
]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("L", LAYERS, ids=lambda L: L.name())
def test_dgrad_requant_sr(cuda_device, fmt, L):
    """dX requantized stochastically into the lower layer's output-gradient
    blocks: bit-exact against the oracle's stochastic quantizer applied to the
    unfused fp32 dX with the same statistic and seed."""
    rng = np.random.default_rng(L.N + L.Cin)
    X = np.maximum(rng.standard_normal(L.x_shape()), 0).astype(np.float32)
    W = (rng.standard_normal(L.w_shape()) * np.sqrt(2 / (L.Cin * L.k * L.k))).astype(np.float32)
    dY = (rng.standard_normal(L.y_shape()) * 0.1).astype(np.float32)
    run = LayerRun(L, fmt, "f32", X, W, dY, cuda_device, check_quant=False)
    dx = run.dgrad()
    dx_np = dx.cpu().numpy()
    stat = float(np.float32(np.abs(dx_np).max() * 1.1))
    for seed in (3, 2 ** 40 + 9):
        out = mq.Packed(fmt, "grad", L.x_shape(), device=cuda_device)
        ain = torch.tensor([stat], device=cuda_device)
        aout = torch.zeros(1, device=cuda_device)
        mq.dgrad(L, run.wq, run.gq, None, rq_out=out, rq_amax_in=ain, rq_amax_out=aout, rq_sr_seed=seed)
        mq.check_device_status()
        ref = oracle.quantize(dx_np, fmt, "grad", "hwcn", amax_in=stat, sr_seed=seed)
        assert_packed_equal(out, ref, f"dgrad SR requant {fmt} {L.name()} seed {seed}")
        assert float(aout.item()) == float(np.abs(dx_np).max())


@pytest.mark.parametrize("L", LAYERS[:2], ids=lambda L: L.name())
def test_fwd_requant_sr(cuda_device, L):
    rng = np.random.default_rng(L.Cout)
    X = np.maximum(rng.standard_normal(L.x_shape()), 0).astype(np.float32)
    W = (rng.standard_normal(L.w_shape()) * np.sqrt(2 / (L.Cin * L.k * L.k))).astype(np.float32)
    run = LayerRun(L, "e2m1", "f32", X, W, np.zeros(L.y_shape(), np.float32), cuda_device, check_quant=False)
    y_np = run.fwd().cpu().numpy()
    stat = float(np.float32(np.abs(y_np).max()))
    out = mq.Packed("e2m1", "act", L.y_shape(), device=cuda_device)
    mq.fwd(L, run.xq, run.wq, None, rq_out=out, rq_amax_in=torch.tensor([stat], device=cuda_device), rq_sr_seed=5)
    mq.check_device_status()
    assert_packed_equal(out, oracle.quantize(y_np, "e2m1", "act", "hwcn", amax_in=stat, sr_seed=5),
                        f"fwd SR requant {L.name()}")
