"""GPU parity of the decoded weight copy (mq_packed.decoded).

The copy is a cache of the packed weight blocks: every value is code * B_scale
(x 1/4 for E4M3 codes), exact in fp16, so it is checked bit for bit against
the oracle's codes and scales.  The convolutions that stage it instead of
decoding the weight blocks on chip must give the same results bit for bit as
the ones that decode: fp32 outputs with torch.equal, fused requantizations
byte for byte.
"""
import numpy as np
import pytest
import torch

import microscaling_quantized_convolution_only_b300 as mq
import oracle
import synthetic as S
from mqtest import LayerRun, to_dev
from synthetic import Layer

pytestmark = pytest.mark.gpu

LAYERS = [
    Layer(8, 16, 8, 8, 16, 3, 1, 1),       # halo kernel, one tile
    Layer(16, 32, 9, 7, 48, 3, 1, 1),      # ragged positions; the last 16 output channels of a 32-wide tile
    Layer(32, 64, 12, 12, 64, 3, 1, 1),    # several tiles
    Layer(16, 32, 10, 14, 48, 3, 2, 1),    # stride 2: forward over column phases, data gradient in quads
    Layer(16, 128, 7, 7, 256, 3, 1, 1),    # deep and small: many chunks, several column tiles
    Layer(8, 16, 6, 6, 24, 5, 1, 2),       # 25 taps (the issue loop without the 3x3 table)
    Layer(8, 24, 10, 10, 16, 1, 2, 0),     # generic kernel: the copy is not used
]
FORMATS = [("e2m1", "e2m1"), ("e2m3", "e2m3"), ("e4m3", "e4m3"), ("e2m1", "e2m3")]   # (X and dY, W)


def _inputs(L, seed):
    rng = np.random.default_rng(seed)
    X = np.maximum(rng.standard_normal(L.x_shape()), 0).astype(np.float32)
    W = (rng.standard_normal(L.w_shape()) * np.sqrt(2 / (L.Cin * L.k * L.k))).astype(np.float32)
    dY = (rng.standard_normal(L.y_shape()) * 0.1).astype(np.float32)
    return X, W, dY


def _expected_decoded(W, fmt):
    """fp16 bits of code * B_scale (x 1/4 for E4M3 codes) per block row, from the oracle."""
    q = oracle.quantize(W, fmt, "weight", "oihw")
    vals = oracle.decode(fmt, oracle.unpack_codes(q))                 # (blocks, 64)
    bs = oracle.decode("e4m3", np.asarray(q["scales"], dtype=np.uint8))
    v = vals * bs[:, None] * (0.25 if fmt == "e4m3" else 1.0)
    h = v.astype(np.float16)
    assert np.array_equal(h.astype(np.float64), v), "decoded values must be exact in fp16"
    return h.view(np.uint16).reshape(-1)


def _with_decoded(run, W, fw, device):
    wqd = mq.Packed(fw, "weight", run.layer.w_shape(), device=device, decoded=True)
    amax = torch.zeros(1, device=device)
    mq.quantize_cbf(to_dev(W, "f32", device), "oihw", wqd, amax_out=amax)
    mq.check_device_status()
    assert torch.equal(wqd.codes, run.wq.codes) and torch.equal(wqd.scales, run.wq.scales)
    return wqd


@pytest.mark.parametrize("fx,fw", FORMATS)
@pytest.mark.parametrize("L", LAYERS, ids=lambda L: L.name())
def test_decoded_copy_matches_oracle_and_decoding(cuda_device, fx, fw, L):
    X, W, dY = _inputs(L, 31 + L.Cout)
    run = LayerRun(L, (fx, fw, fx), "f32", X, W, dY, cuda_device, check_quant=False)
    wqd = _with_decoded(run, W, fw, cuda_device)
    got = wqd.decoded.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, _expected_decoded(W, fw)), "decoded weight copy"
    # forward and data gradient: identical fp32 results with and without the copy
    y_ref, dx_ref = run.fwd(), run.dgrad()
    y = torch.full_like(y_ref, float("nan"))
    mq.fwd(L, run.xq, wqd, y)
    dx = torch.full_like(dx_ref, float("nan"))
    mq.dgrad(L, wqd, run.gq, dx)
    mq.check_device_status()
    assert torch.equal(y, y_ref), "forward with the decoded weight copy"
    assert torch.equal(dx, dx_ref), "data gradient with the decoded weight copy"
    # fused requantizing epilogues: identical packed outputs
    for op, role, shape, ref in (("fwd", "act", L.y_shape(), y_ref), ("dgrad", "grad", L.x_shape(), dx_ref)):
        stat = torch.tensor([float(ref.abs().max().item()) * 1.1], device=cuda_device)
        outs = []
        for w in (run.wq, wqd):
            o = mq.Packed(fx, role, shape, device=cuda_device)
            ao = torch.zeros(1, device=cuda_device)
            if op == "fwd":
                mq.fwd(L, run.xq, w, None, rq_out=o, rq_amax_in=stat, rq_amax_out=ao)
            else:
                mq.dgrad(L, w, run.gq, None, rq_out=o, rq_amax_in=stat, rq_amax_out=ao)
            mq.check_device_status()
            outs.append((o, ao))
        (a, aa), (b, ab) = outs
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales), f"{op} requant codes"
        assert torch.equal(a.s_t, b.s_t) and torch.equal(aa, ab), f"{op} requant T_scale / amax"


def test_weight_decode_rewrites_the_copy(cuda_device):
    """mqconv_weight_decode rebuilds a copy that no longer matches the codes."""
    L = LAYERS[2]
    X, W, dY = _inputs(L, 5)
    run = LayerRun(L, "e2m1", "f32", X, W, dY, cuda_device, check_quant=False)
    wqd = _with_decoded(run, W, "e2m1", cuda_device)
    good = wqd.decoded.clone()
    wqd.decoded.fill_(0x7C)                     # stale contents
    mq.weight_decode(wqd)
    torch.cuda.synchronize()
    assert torch.equal(wqd.decoded, good)


def test_stack_layer_with_decoded_copy(cuda_device):
    """The 56x56 C128 stack layer (batch 64, NVFP4) in the benchmarked plan:
    forward and data gradient identical with and without the copy."""
    wl = S.WORKLOADS[4]
    L = S.scaled_layer(wl.layers[0], N=64)
    X = S.draw_x(wl, 0, L.x_shape())
    W = S.draw_w(wl, 0, L.w_shape())
    dY = S.draw_dy(wl, 0, L.y_shape())
    run = LayerRun(L, wl.fmt, wl.dtype, X, W, dY, cuda_device, check_quant=False)
    wqd = mq.Packed(wl.fmt, "weight", L.w_shape(), device=cuda_device, decoded=True)
    amax = torch.zeros(1, device=cuda_device)
    mq.quantize_cbf(run.Wd, "oihw", wqd, amax_out=amax)
    y_ref, dx_ref = run.fwd(), run.dgrad()
    y = torch.empty_like(y_ref)
    dx = torch.empty_like(dx_ref)
    mq.fwd(L, run.xq, wqd, y)
    mq.dgrad(L, wqd, run.gq, dx)
    mq.check_device_status()
    assert torch.equal(y, y_ref) and torch.equal(dx, dx_ref)


def test_decoded_copy_rejected_on_activations(cuda_device):
    L = LAYERS[0]
    X, W, dY = _inputs(L, 9)
    xq = mq.Packed("e2m1", "act", L.x_shape(), device=cuda_device)
    xq.decoded = torch.empty(1024, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(mq.MQError):
        mq.quantize_cbf(to_dev(X, "f32", cuda_device), "nchw", xq, amax_out=torch.zeros(1, device=cuda_device))
