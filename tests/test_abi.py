"""CPU checks of the C ABI: the library loads, exports every function that
include/mqconv.h declares, and its host-only functions (sizes, planning,
argument validation that returns before any CUDA call) behave.  No kernel is
launched here."""
import ctypes
import os
import re
import subprocess

import pytest

import microscaling_quantized_convolution_only_b300 as mq
from microscaling_quantized_convolution_only_b300 import build as mqbuild
from synthetic import Layer

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mqconv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mqconv_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    mqbuild.build()
    return mq.lib()


def test_header_declares_the_path():
    names = declared_functions()
    for required in ("mqconv_quantize_cbf", "mqconv_fwd", "mqconv_dgrad", "mqconv_wgrad",
                     "mqconv_wgrad_workspace_bytes", "mqconv_device_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", mqbuild.LIB], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (mqconv_\w+)", out.stdout))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for n in declared_functions():
        assert hasattr(lib, n)


def test_abi_version_and_strings(lib):
    assert mq.abi_version() == 3
    assert mq.status_string(0) == "ok"
    assert "multiples of 8" in mq.status_string(2)


@pytest.mark.parametrize("fmt,bb", [("e2m1", 32), ("e2m3", 48), ("e4m3", 64)])
def test_packed_sizes(lib, fmt, bb):
    dims = (64, 128, 7, 9)
    nblk = 8 * 16 * 7 * 9
    assert mq.packed_code_bytes(fmt, dims) == nblk * bb
    assert mq.packed_scale_bytes(dims) == nblk
    assert mq.packed_code_bytes(fmt, (12, 16, 2, 2)) == 0    # batch not a multiple of 8
    assert mq.packed_scale_bytes((8, 0, 2, 2)) == 0


def test_wgrad_workspace_is_split_k_partials(lib):
    L = Layer(256, 128, 56, 56, 128, 3, 1, 1)
    ws = mq.wgrad_workspace_bytes(L)
    assert ws > 0 and ws % (128 * 1152 * 4) == 0
    assert mq.wgrad_workspace_bytes(Layer(12, 16, 8, 8, 16, 3, 1, 1)) == 0


def test_invalid_arguments_rejected_without_launch(lib):
    # null pointers and bad shapes are reported before any CUDA call
    bad = Layer(12, 16, 8, 8, 16, 3, 1, 1)
    d = mq.desc(bad)
    P = mq._Packed
    x = P(4, 0, (ctypes.c_int64 * 4)(12, 16, 8, 8), 16, 16, 16)
    w = P(4, 1, (ctypes.c_int64 * 4)(16, 16, 3, 3), 16, 16, 16)
    assert lib.mqconv_fwd(ctypes.byref(d), ctypes.byref(x), ctypes.byref(w), 16, None, None) == 2
    good = mq.desc(Layer(8, 16, 8, 8, 16, 3, 1, 1))
    assert lib.mqconv_fwd(ctypes.byref(good), None, ctypes.byref(w), 16, None, None) == 1
    assert lib.mqconv_quantize_cbf(None, 0, 0, ctypes.byref(x), None, None, None) == 1
    assert lib.mqconv_device_status(None, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(mq, "_lib", None)
    monkeypatch.setattr(mq, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(mq.MQError):
        mq.lib()


def test_fault_inject_validates_its_arguments(lib):
    """mqconv_test_fault_inject only sets a host-side launch setting."""
    assert lib.mqconv_test_fault_inject(7) == 1               # unknown injection
    assert lib.mqconv_test_fault_inject(1) == 0
    assert lib.mqconv_test_fault_inject(0) == 0               # back to normal operation


def test_decoded_weight_copy_sizes_and_checks(lib):
    """The decoded weight copy: 128 bytes per block; a copy on a tensor of another
    role, a misaligned copy and a decode request without one are argument errors,
    reported before any CUDA call."""
    assert mq.weight_decoded_bytes((64, 128, 3, 3)) == 8 * 16 * 9 * 128
    assert mq.weight_decoded_bytes((12, 16, 3, 3)) == 0
    P = mq._Packed
    good = mq.desc(Layer(8, 16, 8, 8, 16, 3, 1, 1))
    x_dec = P(4, 0, (ctypes.c_int64 * 4)(8, 16, 8, 8), 16, 16, 16, 16)       # ACT with a decoded copy
    x = P(4, 0, (ctypes.c_int64 * 4)(8, 16, 8, 8), 16, 16, 16, None)
    w = P(4, 1, (ctypes.c_int64 * 4)(16, 16, 3, 3), 16, 16, 16, None)
    w_mis = P(4, 1, (ctypes.c_int64 * 4)(16, 16, 3, 3), 16, 16, 16, 24)     # decoded not 16-byte aligned
    assert lib.mqconv_fwd(ctypes.byref(good), ctypes.byref(x_dec), ctypes.byref(w), 16, None, None) == 1
    assert lib.mqconv_fwd(ctypes.byref(good), ctypes.byref(x), ctypes.byref(w_mis), 16, None, None) == 3
    assert lib.mqconv_weight_decode(ctypes.byref(w), None) == 1                # no decoded copy
    assert lib.mqconv_weight_decode(ctypes.byref(x_dec), None) == 1            # not a weight tensor
    assert lib.mqconv_weight_decode(ctypes.byref(w_mis), None) == 3
