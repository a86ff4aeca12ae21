"""Seeded synthetic inputs and the layer shapes of the five workloads.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It draws random numbers and describes shapes; it holds none of the
quantization or convolution arithmetic.

Random stream: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) in counter form -- output i of a stream with
seed s is mix(s + (i + 1) * 0x9E3779B97F4A7C15) -- mapped to a uniform in
(0, 1] by its top 53 bits, and to standard normals by the Box-Muller transform
(pairs (2j, 2j+1) of uniforms give normals 2j and 2j+1).

Distributions follow the workload descriptions: activations ReLU(N(0, 1)),
weights Kaiming-normal N(0, 2 / (C_in * Kh * Kw)), output gradients N(0, v)
with v the variance (1e-2 or 1e-3).  bf16 workloads round the fp32 draw to
bf16 with round-to-nearest-even.  Seeds are 1000 * config + 10 * layer +
{X: 0, W: 1, dY: 2}.

The layer shapes are those of the networks the MicroQonv paper trains
(ResNet-32 on CIFAR-100, ResNet-18 on ImageNet, YOLOv8n at 640 px; MicroQonv,
§IV-D and §IV-E); no dataset is used, only the shapes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform(seed: int, count: int, start: int = 0) -> np.ndarray:
    """Uniforms in (0, 1] (float64): elements start .. start+count-1 of stream `seed`."""
    out = np.empty(count, dtype=np.float64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, count, _CHUNK):
            hi = min(count, lo + _CHUNK)
            idx = np.arange(start + lo + 1, start + hi + 1, dtype=np.uint64)
            z = _mix(s + idx * GOLDEN_GAMMA)
            out[lo:hi] = ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    return out


def normal(seed: int, count: int) -> np.ndarray:
    """`count` standard normals (float64) from stream `seed` via Box-Muller."""
    pairs = (count + 1) // 2
    out = np.empty(2 * pairs, dtype=np.float64)
    for lo in range(0, pairs, _CHUNK):
        hi = min(pairs, lo + _CHUNK)
        u = uniform(seed, 2 * (hi - lo), start=2 * lo)
        r = np.sqrt(-2.0 * np.log(u[0::2]))
        t = 2.0 * math.pi * u[1::2]
        out[2 * lo:2 * hi:2] = r * np.cos(t)
        out[2 * lo + 1:2 * hi:2] = r * np.sin(t)
    return out[:count]


def to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returned widened to float32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    r = (b + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


@dataclasses.dataclass(frozen=True)
class Layer:
    N: int
    Cin: int
    H: int
    W: int
    Cout: int
    k: int
    stride: int
    pad: int

    @property
    def Ho(self) -> int:
        return (self.H + 2 * self.pad - self.k) // self.stride + 1

    @property
    def Wo(self) -> int:
        return (self.W + 2 * self.pad - self.k) // self.stride + 1

    @property
    def flops(self) -> int:
        """Dense conv FLOPs of one GEMM (fwd, dgrad and wgrad share it)."""
        return 2 * self.N * self.Cout * self.Ho * self.Wo * self.Cin * self.k * self.k

    def x_shape(self):
        return (self.N, self.Cin, self.H, self.W)

    def w_shape(self):
        return (self.Cout, self.Cin, self.k, self.k)

    def y_shape(self):
        return (self.N, self.Cout, self.Ho, self.Wo)

    def name(self) -> str:
        return (f"N{self.N}_{self.H}x{self.W}_C{self.Cin}-{self.Cout}"
                f"_k{self.k}s{self.stride}p{self.pad}")


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    name: str
    layers: List[Layer]
    fmt: str            # element format of every tensor: "e2m1" | "e2m3" | "e4m3"
    dtype: str          # input dtype of X, W, dY: "f32" | "bf16"
    dy_var: float       # variance of the output-gradient draw
    chained: bool = False

    def seed(self, layer: int, tensor: str) -> int:
        return 1000 * self.index + 10 * layer + {"X": 0, "W": 1, "dY": 2}[tensor]


def _r32(H, ci, co, s):
    return Layer(128, ci, H, H, co, 3, s, 1)


def _r18(H, ci, co, k, s, p):
    return Layer(64, ci, H, H, co, k, s, p)


def _yolo(H, ci, co, k, s, p):
    return Layer(16, ci, H, H, co, k, s, p)


WORKLOADS = {
    0: Workload(0, "tiny-3x3", [Layer(8, 16, 8, 8, 16, 3, 1, 1)], "e2m1", "f32", 1e-2),
    1: Workload(1, "resnet32-cifar", [
        _r32(32, 16, 16, 1), _r32(16, 32, 32, 1), _r32(8, 64, 64, 1),
        _r32(32, 16, 32, 2), _r32(16, 32, 64, 2)], "e2m1", "f32", 1e-2),
    2: Workload(2, "resnet18-224", [
        _r18(56, 64, 64, 3, 1, 1), _r18(28, 128, 128, 3, 1, 1),
        _r18(14, 256, 256, 3, 1, 1), _r18(7, 512, 512, 3, 1, 1),
        _r18(56, 64, 128, 3, 2, 1), _r18(28, 128, 256, 3, 2, 1),
        _r18(14, 256, 512, 3, 2, 1),
        _r18(56, 64, 128, 1, 2, 0), _r18(28, 128, 256, 1, 2, 0),
        _r18(14, 256, 512, 1, 2, 0)], "e2m1", "bf16", 1e-3),
    3: Workload(3, "yolov8n-640-fp8", [
        _yolo(320, 16, 32, 3, 2, 1), _yolo(160, 32, 32, 3, 1, 1),
        _yolo(160, 32, 64, 3, 2, 1), _yolo(80, 64, 64, 3, 1, 1),
        _yolo(40, 128, 128, 3, 1, 1), _yolo(20, 256, 256, 3, 1, 1),
        _yolo(80, 64, 32, 1, 1, 0), _yolo(40, 128, 64, 1, 1, 0)], "e4m3", "f32", 1e-2),
    4: Workload(4, "stack4-56x56-c128-nvfp4", [Layer(256, 128, 56, 56, 128, 3, 1, 1)] * 4,
                "e2m1", "bf16", 1e-3, chained=True),
    5: Workload(4, "stack4-56x56-c128-fp6", [Layer(256, 128, 56, 56, 128, 3, 1, 1)] * 4,
                "e2m3", "bf16", 1e-3, chained=True),
}


def _finish(x: np.ndarray, dtype: str) -> np.ndarray:
    x = x.astype(np.float32)
    return to_bf16_rne(x) if dtype == "bf16" else x


def draw_x(wl: Workload, layer: int, shape=None) -> np.ndarray:
    """ReLU(N(0,1)) activations, NCHW float32 (bf16-valued for bf16 workloads)."""
    shape = shape or wl.layers[layer].x_shape()
    n = normal(wl.seed(layer, "X"), int(np.prod(shape)))
    return _finish(np.maximum(n, 0.0), wl.dtype).reshape(shape)


def draw_w(wl: Workload, layer: int, shape=None) -> np.ndarray:
    """Kaiming-normal weights N(0, 2/(Cin*Kh*Kw)), OIHW float32."""
    shape = shape or wl.layers[layer].w_shape()
    std = math.sqrt(2.0 / (shape[1] * shape[2] * shape[3]))
    n = normal(wl.seed(layer, "W"), int(np.prod(shape)))
    return _finish(n * std, wl.dtype).reshape(shape)


def draw_dy(wl: Workload, layer: int, shape=None) -> np.ndarray:
    """Output gradients N(0, dy_var), NCHW (N, Cout, Ho, Wo) float32."""
    shape = shape or wl.layers[layer].y_shape()
    n = normal(wl.seed(layer, "dY"), int(np.prod(shape)))
    return _finish(n * math.sqrt(wl.dy_var), wl.dtype).reshape(shape)


def scaled_layer(layer: Layer, N: Optional[int] = None, H: Optional[int] = None) -> Layer:
    """Same layer with a smaller batch and/or spatial size (for CPU-sized parity cases)."""
    return dataclasses.replace(layer, N=N or layer.N, H=H or layer.H, W=H or layer.W)
