"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding, and compare against the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import microscaling_quantized_convolution_only_b300 as mq
import oracle

# conv tolerance: |gpu - ref| <= RTOL_ABS * sum|a*b| + ATOL per element, and
# relative L2 error <= RTOL_L2 per tensor.
RTOL_ABS = 1e-5
ATOL = 1e-7
RTOL_L2 = 1e-5


def to_dev(x: np.ndarray, dtype: str, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)   # exact: the values are already bf16-representable
    return t.to(device)


def gpu_quantize(x_dev: torch.Tensor, fmt: str, role: str, layout: str, dims, amax_in=None):
    """Quantize on the GPU; returns (Packed, measured amax as float)."""
    p = mq.Packed(fmt, role, dims, device=x_dev.device)
    amax_out = torch.zeros(1, dtype=torch.float32, device=x_dev.device)
    ain = None
    if amax_in is not None:
        ain = torch.tensor([amax_in], dtype=torch.float32, device=x_dev.device)
    mq.quantize_cbf(x_dev, layout, p, amax_in=ain, amax_out=amax_out)
    mq.check_device_status()
    return p, float(amax_out.item())


def packed_to_oracle(p: "mq.Packed") -> dict:
    return {"codes": p.codes.cpu().numpy(), "scales": p.scales.cpu().numpy(), "s_t": float(p.s_t.item()),
            "fmt": p.fmt, "role": p.role, "dims": p.dims}


def assert_packed_equal(p: "mq.Packed", ref: dict, what: str = ""):
    codes = p.codes.cpu().numpy()
    scales = p.scales.cpu().numpy()
    st = float(p.s_t.item())
    assert st == ref["s_t"], f"{what}: T_scale {st!r} != {ref['s_t']!r}"
    bad_s = np.flatnonzero(scales != ref["scales"])
    assert bad_s.size == 0, f"{what}: {bad_s.size} scale bytes differ, first at block {bad_s[:5]}"
    bad_c = np.flatnonzero(codes != ref["codes"])
    assert bad_c.size == 0, f"{what}: {bad_c.size} code bytes differ, first at byte {bad_c[:5]}"


def check_close(gpu: np.ndarray, ref: np.ndarray, refabs: np.ndarray, what: str):
    gpu = np.asarray(gpu, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = RTOL_ABS * refabs + ATOL
    bad = np.flatnonzero(err > bound)
    assert bad.size == 0, (f"{what}: {bad.size}/{err.size} elements out of tolerance; worst "
                           f"err/bound {np.max(err / bound):.3g} at {np.argmax(err / bound)}")
    rel = np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= RTOL_L2, f"{what}: relative L2 error {rel:.3g} > {RTOL_L2}"
    return float(np.max(err / bound)), float(rel)


def hwcn_to_nchw(t: torch.Tensor) -> np.ndarray:
    """[H][W][C][N] device tensor -> NCHW numpy."""
    return t.permute(3, 2, 0, 1).contiguous().cpu().numpy()


class LayerRun:
    """Quantize X, W, dY of one layer on the GPU (checked bit-exact against the
    oracle) and run fwd/dgrad/wgrad."""

    def __init__(self, layer, fmt, dtype, X, W, dY, device, check_quant=True):
        # fmt: one element format for X, W and dY, or a (X, W, dY) triple
        # (MicroQonv+: each tensor in its own format)
        self.layer, self.fmt, self.dtype, self.device = layer, fmt, dtype, device
        fx, fw, fg = fmt if isinstance(fmt, tuple) else (fmt, fmt, fmt)
        L = layer
        self.Xd, self.Wd, self.dYd = (to_dev(a, dtype, device) for a in (X, W, dY))
        self.xq, _ = gpu_quantize(self.Xd, fx, "act", "nchw", L.x_shape())
        self.wq, _ = gpu_quantize(self.Wd, fw, "weight", "oihw", L.w_shape())
        self.gq, _ = gpu_quantize(self.dYd, fg, "grad", "nchw", L.y_shape())
        if check_quant:
            for p, a, f, role, lay in ((self.xq, X, fx, "act", "nchw"), (self.wq, W, fw, "weight", "oihw"),
                                       (self.gq, dY, fg, "grad", "nchw")):
                assert_packed_equal(p, oracle.quantize(a, f, role, lay), f"{role} quantization")

    def fwd(self):
        L = self.layer
        y = torch.empty((L.Ho, L.Wo, L.Cout, L.N), dtype=torch.float32, device=self.device)
        mq.fwd(L, self.xq, self.wq, y)
        mq.check_device_status()
        return y

    def dgrad(self):
        L = self.layer
        dx = torch.empty((L.H, L.W, L.Cin, L.N), dtype=torch.float32, device=self.device)
        mq.dgrad(L, self.wq, self.gq, dx)
        mq.check_device_status()
        return dx

    def wgrad(self):
        L = self.layer
        dw = torch.empty(L.w_shape(), dtype=torch.float32, device=self.device)
        ws = torch.empty(max(16, mq.wgrad_workspace_bytes(L)), dtype=torch.uint8, device=self.device)
        mq.wgrad(L, self.gq, self.xq, dw, ws)
        mq.check_device_status()
        return dw

    def oracle_operands(self):
        return (oracle.dequantize(packed_to_oracle(self.xq)), oracle.dequantize(packed_to_oracle(self.wq)),
                oracle.dequantize(packed_to_oracle(self.gq)))
