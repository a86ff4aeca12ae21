"""Python binding of libmqconv (the C ABI in include/mqconv.h).

Argument marshalling only: every step of quantization and convolution runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.  There
is no fallback: if libmqconv.so is missing or a call fails, this module raises.

Entry points mirror the C names: quantize_cbf (and, with sr_seed,
quantize_cbf_sr), fwd, dgrad (and, with rq_out, dgrad_requant), wgrad,
wgrad_noalloc, wgrad_workspace_bytes, packed_code_bytes, packed_scale_bytes,
device_status, test_fault_inject.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

LIB_PATH = _build.LIB

FMT = {"e2m1": 4, "e2m3": 6, "e4m3": 8}
ROLE = {"act": 0, "weight": 1, "grad": 2}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
LAYOUT = {"nchw": 0, "hwcn": 1, "oihw": 2}
ERR_BITS = {4: "non-finite input", 5: "bounded wait expired"}


class MQError(RuntimeError):
    pass


class _Packed(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("role", ctypes.c_int32), ("dims", ctypes.c_int64 * 4),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("s_t", ctypes.c_void_p),
                ("decoded", ctypes.c_void_p)]


class _Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("N", "Cin", "H", "W", "Cout", "Kh", "Kw", "stride", "pad")]


class _Requant(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("amax_in", ctypes.c_void_p), ("out", ctypes.POINTER(_Packed)),
                ("amax_out", ctypes.c_void_p), ("rounding", ctypes.c_int32), ("sr_seed", ctypes.c_uint64)]


def _requant(rq_out, rq_amax_in, rq_amax_out, sr_seed):
    out_c = rq_out.c()
    rq = _Requant(FMT[rq_out.fmt], _ptr(rq_amax_in), ctypes.pointer(out_c), _ptr(rq_amax_out),
                  0 if sr_seed is None else 1, 0 if sr_seed is None else sr_seed & 0xFFFFFFFFFFFFFFFF)
    rq._keep = out_c
    return rq


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmqconv.so (built by __graft_entry__.build() / build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MQError(f"libmqconv.so not built ({LIB_PATH}); run build.py")
        L = ctypes.CDLL(LIB_PATH)
        P, i32 = ctypes.c_void_p, ctypes.c_int32
        L.mqconv_abi_version.restype = i32
        L.mqconv_status_string.argtypes = [i32]
        L.mqconv_status_string.restype = ctypes.c_char_p
        L.mqconv_packed_code_bytes.argtypes = [i32, P]
        L.mqconv_packed_code_bytes.restype = ctypes.c_size_t
        L.mqconv_packed_scale_bytes.argtypes = [P]
        L.mqconv_packed_scale_bytes.restype = ctypes.c_size_t
        L.mqconv_weight_decoded_bytes.argtypes = [P]
        L.mqconv_weight_decoded_bytes.restype = ctypes.c_size_t
        L.mqconv_weight_decode.argtypes = [ctypes.POINTER(_Packed), P]
        L.mqconv_quantize_cbf.argtypes = [P, i32, i32, ctypes.POINTER(_Packed), P, P, P]
        L.mqconv_quantize_cbf_sr.argtypes = [P, i32, i32, ctypes.POINTER(_Packed), P, P, ctypes.c_uint64, P]
        L.mqconv_fwd.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Packed), ctypes.POINTER(_Packed), P,
                                 ctypes.POINTER(_Requant), P]
        L.mqconv_dgrad.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Packed), ctypes.POINTER(_Packed), P, P]
        L.mqconv_dgrad_requant.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Packed), ctypes.POINTER(_Packed),
                                           P, ctypes.POINTER(_Requant), P]
        L.mqconv_wgrad_workspace_bytes.argtypes = [ctypes.POINTER(_Desc)]
        L.mqconv_wgrad_workspace_bytes.restype = ctypes.c_size_t
        L.mqconv_wgrad.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Packed), ctypes.POINTER(_Packed), P, P,
                                   ctypes.c_size_t, P]
        L.mqconv_device_status.argtypes = [P, ctypes.POINTER(i32)]
        L.mqconv_wgrad_noalloc.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(_Packed), ctypes.POINTER(_Packed), P,
                                           P]
        L.mqconv_test_fault_inject.argtypes = [i32]
        for f in ("mqconv_quantize_cbf", "mqconv_quantize_cbf_sr", "mqconv_fwd", "mqconv_dgrad", "mqconv_dgrad_requant", "mqconv_wgrad",
                  "mqconv_device_status", "mqconv_wgrad_noalloc", "mqconv_test_fault_inject", "mqconv_weight_decode"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def abi_version() -> int:
    return int(lib().mqconv_abi_version())


def status_string(code: int) -> str:
    return lib().mqconv_status_string(code).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise MQError(f"{what}: {status_string(rc)} (status {rc})")


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dims(d: Sequence[int]):
    return (ctypes.c_int64 * 4)(*[int(v) for v in d])


def packed_code_bytes(fmt: str, dims: Sequence[int]) -> int:
    return int(lib().mqconv_packed_code_bytes(FMT[fmt], ctypes.cast(_dims(dims), ctypes.c_void_p)))


def packed_scale_bytes(dims: Sequence[int]) -> int:
    return int(lib().mqconv_packed_scale_bytes(ctypes.cast(_dims(dims), ctypes.c_void_p)))


def weight_decoded_bytes(dims: Sequence[int]) -> int:
    return int(lib().mqconv_weight_decoded_bytes(ctypes.cast(_dims(dims), ctypes.c_void_p)))


class Packed:
    """A packed 8x8-block tensor whose buffers are torch device tensors.

    dims: act/grad (N, C, H, W); weight (Cout, Cin, Kh, Kw).  decoded (weights
    only): True to allocate the decoded fp16 copy (mq_packed.decoded), or a
    uint8 device tensor of weight_decoded_bytes(dims) bytes to use as it."""

    def __init__(self, fmt: str, role: str, dims: Sequence[int], device="cuda", codes=None, scales=None, s_t=None,
                 decoded=None):
        self.fmt, self.role, self.dims = fmt, role, tuple(int(v) for v in dims)
        nc, ns = packed_code_bytes(fmt, self.dims), packed_scale_bytes(self.dims)
        if nc == 0:
            raise MQError(f"invalid packed dims {self.dims} for {fmt}")
        self.codes = codes if codes is not None else torch.empty(nc, dtype=torch.uint8, device=device)
        self.scales = scales if scales is not None else torch.empty(ns, dtype=torch.uint8, device=device)
        self.s_t = s_t if s_t is not None else torch.zeros(1, dtype=torch.float32, device=device)
        if decoded is True:
            decoded = torch.empty(weight_decoded_bytes(self.dims), dtype=torch.uint8, device=device)
        self.decoded = decoded if decoded is not None and decoded is not False else None

    def c(self) -> _Packed:
        return _Packed(FMT[self.fmt], ROLE[self.role], _dims(self.dims), self.codes.data_ptr(),
                       self.scales.data_ptr(), self.s_t.data_ptr(),
                       None if self.decoded is None else self.decoded.data_ptr())


def weight_decode(wq: Packed, stream=None) -> None:
    """mqconv_weight_decode: rewrite wq.decoded from wq's codes and scales."""
    c = wq.c()
    _check(lib().mqconv_weight_decode(ctypes.byref(c), _stream(stream)), "mqconv_weight_decode")


def desc(layer) -> _Desc:
    """mq_conv_desc from any object with N, Cin, H, W, Cout, k (or Kh, Kw), stride, pad."""
    kh = getattr(layer, "Kh", None) or layer.k
    kw = getattr(layer, "Kw", None) or layer.k
    return _Desc(layer.N, layer.Cin, layer.H, layer.W, layer.Cout, kh, kw, layer.stride, layer.pad)


def quantize_cbf(src: torch.Tensor, layout: str, dst: Packed, amax_in: Optional[torch.Tensor] = None,
                 amax_out: Optional[torch.Tensor] = None, stream=None, sr_seed: Optional[int] = None) -> None:
    """mqconv_quantize_cbf: quantize `src` (fp32/bf16, dense in `layout`) once into `dst`;
    with sr_seed, mqconv_quantize_cbf_sr (stochastic element codes, Philox key sr_seed)."""
    if not src.is_contiguous():
        raise MQError("src must be contiguous")
    c = dst.c()
    if sr_seed is None:
        rc = lib().mqconv_quantize_cbf(src.data_ptr(), DTYPE[src.dtype], LAYOUT[layout], ctypes.byref(c),
                                       _ptr(amax_in), _ptr(amax_out), _stream(stream))
        _check(rc, "mqconv_quantize_cbf")
    else:
        rc = lib().mqconv_quantize_cbf_sr(src.data_ptr(), DTYPE[src.dtype], LAYOUT[layout], ctypes.byref(c),
                                          _ptr(amax_in), _ptr(amax_out), ctypes.c_uint64(sr_seed & 0xFFFFFFFFFFFFFFFF),
                                          _stream(stream))
        _check(rc, "mqconv_quantize_cbf_sr")


def fwd(layer, xq: Packed, wq: Packed, y: Optional[torch.Tensor], rq_out: Optional[Packed] = None,
        rq_amax_in: Optional[torch.Tensor] = None, rq_amax_out: Optional[torch.Tensor] = None, stream=None,
        rq_sr_seed: Optional[int] = None) -> None:
    """mqconv_fwd: Y (fp32, [Ho][Wo][Cout][N]) and/or the fused requantization of Y into rq_out
    (stochastic element codes with Philox key rq_sr_seed when given)."""
    d, x, w = desc(layer), xq.c(), wq.c()
    rq_p = None
    if rq_out is not None:
        rq = _requant(rq_out, rq_amax_in, rq_amax_out, rq_sr_seed)
        rq_p = ctypes.byref(rq)
    rc = lib().mqconv_fwd(ctypes.byref(d), ctypes.byref(x), ctypes.byref(w), _ptr(y), rq_p, _stream(stream))
    _check(rc, "mqconv_fwd")


def dgrad(layer, wq: Packed, dyq: Packed, dx: Optional[torch.Tensor], rq_out: Optional[Packed] = None,
          rq_amax_in: Optional[torch.Tensor] = None, rq_amax_out: Optional[torch.Tensor] = None, stream=None,
          rq_sr_seed: Optional[int] = None) -> None:
    """mqconv_dgrad: dX (fp32, [H][W][Cin][N]); with rq_out, mqconv_dgrad_requant: dX (optional) and its
    fused requantization into rq_out (role grad, dims (N, Cin, H, W); stochastic element codes with Philox
    key rq_sr_seed when given)."""
    d, w, g = desc(layer), wq.c(), dyq.c()
    if rq_out is None:
        rc = lib().mqconv_dgrad(ctypes.byref(d), ctypes.byref(w), ctypes.byref(g), _ptr(dx), _stream(stream))
        _check(rc, "mqconv_dgrad")
        return
    rq = _requant(rq_out, rq_amax_in, rq_amax_out, rq_sr_seed)
    rc = lib().mqconv_dgrad_requant(ctypes.byref(d), ctypes.byref(w), ctypes.byref(g), _ptr(dx), ctypes.byref(rq),
                                    _stream(stream))
    _check(rc, "mqconv_dgrad_requant")


def wgrad_workspace_bytes(layer) -> int:
    d = desc(layer)
    return int(lib().mqconv_wgrad_workspace_bytes(ctypes.byref(d)))


def wgrad(layer, dyq: Packed, xq: Packed, dw: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """mqconv_wgrad: dW (fp32, [Cout][Cin][Kh][Kw]); workspace >= wgrad_workspace_bytes(layer) bytes."""
    d, g, x = desc(layer), dyq.c(), xq.c()
    rc = lib().mqconv_wgrad(ctypes.byref(d), ctypes.byref(g), ctypes.byref(x), _ptr(dw), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mqconv_wgrad")


def wgrad_noalloc(layer, dyq: Packed, xq: Packed, dw: torch.Tensor, stream=None) -> None:
    """mqconv_wgrad_noalloc: dW like wgrad(), with no workspace and no device
    allocation anywhere (the partial sums use the library's built-in scratch)."""
    d, g, x = desc(layer), dyq.c(), xq.c()
    rc = lib().mqconv_wgrad_noalloc(ctypes.byref(d), ctypes.byref(g), ctypes.byref(x), _ptr(dw), _stream(stream))
    _check(rc, "mqconv_wgrad_noalloc")


INJECT = {"none": 0, "withhold_acc_release": 1}


def test_fault_inject(what: str = "none") -> None:
    """mqconv_test_fault_inject: test support for the failure detection (see
    include/mqconv.h).  "none" restores normal operation."""
    _check(lib().mqconv_test_fault_inject(INJECT[what]), "mqconv_test_fault_inject")


def device_status(stream=None) -> int:
    """mqconv_device_status: synchronize, read and clear the device status word."""
    v = ctypes.c_int32(0)
    _check(lib().mqconv_device_status(_stream(stream), ctypes.byref(v)), "mqconv_device_status")
    return int(v.value)


def check_device_status(stream=None) -> None:
    v = device_status(stream)
    if v:
        bits = [name for b, name in ERR_BITS.items() if v & (1 << b)]
        raise MQError(f"device status {v:#x}: {', '.join(bits) or 'unknown'}")
