"""CPU oracle for MicroQonv quantize-once convolution -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's cpu_baseline/reference
legs may import this package.  It shares no code with the CUDA path: the
arithmetic lives in ``mqoracle.c`` (plain C, fp64), loaded here with ctypes,
plus the instrumented naive flows below (plain numpy) that count how often each
activation is quantized under the flows the paper compares against.

Sources (paper "MicroQonv: Reshaping Convolution Tensors for Efficient
Microscaling in Training and Inference"):
  * quantizer: §III-A (Microscaling quantization), §IV-B (square 8x8 blocks)
  * convolutions: §II-A, §II-C, §IV-A (the three GEMMs on the CBF layout)
  * naive flows and their counts: §III-C (Limitations of related work),
    §IV-C and Table I.

Parity status: every function here is pinned by tests/test_oracle_*.py against
closed forms, brute force, independent library routines (torch float8 casts,
torch fp64 convolutions) or the values printed in Table I.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mqoracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FORMATS = {"e2m1": 4, "e2m3": 6, "e4m3": 8}
ROLES = {"act": 0, "weight": 1, "grad": 2}
LAYOUTS = {"nchw": 0, "hwcn": 1, "oihw": 2}
BLOCK_BYTES = {"e2m1": 32, "e2m3": 48, "e4m3": 64}

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (fp contraction off, OpenMP on)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", "-Wextra", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        L.orc_format_grid.argtypes = [ctypes.c_int, P, P]
        L.orc_round.argtypes = [ctypes.c_int, P, i64, P]
        L.orc_decode.argtypes = [ctypes.c_int, P, i64, P]
        L.orc_tensor_scale.argtypes = [ctypes.c_int, ctypes.c_float]
        L.orc_tensor_scale.restype = ctypes.c_float
        L.orc_num_blocks.argtypes = [ctypes.c_int, P]
        L.orc_num_blocks.restype = i64
        L.orc_quantize.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P]
        L.orc_quantize_sr.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_uint64,
                                      P, P, P, P]
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_philox4x32_10.restype = None
        L.orc_dequantize.argtypes = [P, P, ctypes.c_float, ctypes.c_int, ctypes.c_int, P, P]
        for name in ("orc_conv_fwd", "orc_conv_dgrad", "orc_conv_wgrad"):
            getattr(L, name).argtypes = [P, P, P, P, P]
            getattr(L, name).restype = None
        for name in ("orc_conv_fwd_at", "orc_conv_dgrad_at", "orc_conv_wgrad_at"):
            getattr(L, name).argtypes = [P, P, P, P, i64, P, P]
            getattr(L, name).restype = None
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc == 2:
        raise FloatingPointError(f"{what}: non-finite input")
    if rc != 0:
        raise ValueError(f"{what}: invalid argument (code {rc})")


# ------------------------------------------------------------------ formats

def format_grid(fmt: str) -> np.ndarray:
    """Finite non-negative values of an element format, indexed by magnitude code."""
    out = np.zeros(256, dtype=np.float64)
    cnt = ctypes.c_int(0)
    _check(lib().orc_format_grid(FORMATS[fmt], _p(out), ctypes.byref(cnt)), "format_grid")
    return out[:cnt.value].copy()


def round_codes(fmt: str, q: np.ndarray) -> np.ndarray:
    """Nearest code (ties to even, satfinite, sign kept) of each fp64 value."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.zeros(q.shape, dtype=np.uint8)
    _check(lib().orc_round(FORMATS[fmt], _p(q), q.size, _p(out)), "round")
    return out


def decode(fmt: str, codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(codes.shape, dtype=np.float64)
    _check(lib().orc_decode(FORMATS[fmt], _p(codes), codes.size, _p(out)), "decode")
    return out


def tensor_scale(fmt: str, amax: float) -> float:
    return float(lib().orc_tensor_scale(FORMATS[fmt], ctypes.c_float(amax)))


# ---------------------------------------------------------------- quantizer

def packed_sizes(fmt: str, role: str, dims) -> Dict[str, int]:
    d = np.asarray(dims, dtype=np.int64)
    nb = int(lib().orc_num_blocks(ROLES[role], _p(d)))
    return {"blocks": nb, "code_bytes": nb * BLOCK_BYTES[fmt], "scale_bytes": nb}


def quantize(src: np.ndarray, fmt: str, role: str, layout: str,
             amax_in: Optional[float] = None, sr_seed: Optional[int] = None) -> Dict[str, object]:
    """Quantize a dense fp32 tensor once into packed 8x8 blocks.

    dims are read from the logical shape: act/grad (N, C, H, W) whatever the
    memory layout; weight (Cout, Cin, Kh, Kw).  For layout "hwcn" `src` must
    have memory shape (H, W, C, N).  sr_seed: None for round-to-nearest
    element codes, else stochastic rounding with that 64-bit Philox key
    (mqoracle.c, "stochastic rounding").
    """
    src = np.ascontiguousarray(src, dtype=np.float32)
    if layout == "hwcn":
        H, W, C, N = src.shape
        dims = (N, C, H, W)
    else:
        dims = src.shape
    d = np.asarray(dims, dtype=np.int64)
    sz = packed_sizes(fmt, role, dims)
    codes = np.zeros(sz["code_bytes"], dtype=np.uint8)
    scales = np.zeros(sz["scale_bytes"], dtype=np.uint8)
    s_t = ctypes.c_float(0.0)
    amax = ctypes.c_float(0.0)
    ain = ctypes.c_float(amax_in) if amax_in is not None else None
    if sr_seed is None:
        rc = lib().orc_quantize(_p(src), LAYOUTS[layout], ROLES[role], FORMATS[fmt], _p(d),
                                ctypes.byref(ain) if ain is not None else None,
                                _p(codes), _p(scales), ctypes.byref(s_t), ctypes.byref(amax))
    else:
        rc = lib().orc_quantize_sr(_p(src), LAYOUTS[layout], ROLES[role], FORMATS[fmt], _p(d),
                                   ctypes.byref(ain) if ain is not None else None,
                                   ctypes.c_uint64(sr_seed & 0xFFFFFFFFFFFFFFFF),
                                   _p(codes), _p(scales), ctypes.byref(s_t), ctypes.byref(amax))
    _check(rc, "quantize")
    return {"codes": codes, "scales": scales, "s_t": float(s_t.value), "amax": float(amax.value),
            "fmt": fmt, "role": role, "dims": tuple(int(x) for x in dims)}


def philox4x32_10(ctr, key) -> np.ndarray:
    """The four 32-bit output words of Philox4x32-10 for a counter (4 words)
    and key (2 words)."""
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def dequantize(q: Dict[str, object]) -> np.ndarray:
    """Fake-quantized fp64 tensor: NCHW for act/grad, OIHW for weight."""
    dims = q["dims"]
    d = np.asarray(dims, dtype=np.int64)
    out = np.zeros(dims, dtype=np.float64)
    rc = lib().orc_dequantize(_p(q["codes"]), _p(q["scales"]), ctypes.c_float(q["s_t"]),
                              ROLES[q["role"]], FORMATS[q["fmt"]], _p(d), _p(out))
    _check(rc, "dequantize")
    return out


# ------------------------------------------------------------- convolution

def _geom(layer) -> np.ndarray:
    return np.asarray([layer.N, layer.Cin, layer.H, layer.W, layer.Cout,
                       layer.k, layer.k, layer.stride, layer.pad], dtype=np.int64)


def conv_fwd(X: np.ndarray, W: np.ndarray, layer):
    """Y (N, Cout, Ho, Wo) and sum|a*b| per element, fp64."""
    X = np.ascontiguousarray(X, dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.float64)
    Y = np.zeros(layer.y_shape(), dtype=np.float64)
    Ya = np.zeros_like(Y)
    lib().orc_conv_fwd(_p(X), _p(W), _p(_geom(layer)), _p(Y), _p(Ya))
    return Y, Ya


def conv_dgrad(W: np.ndarray, dY: np.ndarray, layer):
    """dX (N, Cin, H, W) and sum|a*b| per element, fp64."""
    W = np.ascontiguousarray(W, dtype=np.float64)
    dY = np.ascontiguousarray(dY, dtype=np.float64)
    dX = np.zeros(layer.x_shape(), dtype=np.float64)
    dXa = np.zeros_like(dX)
    lib().orc_conv_dgrad(_p(W), _p(dY), _p(_geom(layer)), _p(dX), _p(dXa))
    return dX, dXa


def conv_wgrad(dY: np.ndarray, X: np.ndarray, layer):
    """dW (Cout, Cin, Kh, Kw) and sum|a*b| per element, fp64."""
    dY = np.ascontiguousarray(dY, dtype=np.float64)
    X = np.ascontiguousarray(X, dtype=np.float64)
    dW = np.zeros(layer.w_shape(), dtype=np.float64)
    dWa = np.zeros_like(dW)
    lib().orc_conv_wgrad(_p(dY), _p(X), _p(_geom(layer)), _p(dW), _p(dWa))
    return dW, dWa


def _sampled(fn, A, B, layer, idx):
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.zeros(idx.size, dtype=np.float64)
    outa = np.zeros(idx.size, dtype=np.float64)
    fn(_p(A), _p(B), _p(_geom(layer)), _p(idx), idx.size, _p(out), _p(outa))
    return out, outa


def conv_fwd_at(X, W, layer, idx):
    """Y at flat NCHW indices `idx` (Y shape (N, Cout, Ho, Wo))."""
    return _sampled(lib().orc_conv_fwd_at, X, W, layer, idx)


def conv_dgrad_at(W, dY, layer, idx):
    """dX at flat NCHW indices `idx`."""
    return _sampled(lib().orc_conv_dgrad_at, W, dY, layer, idx)


def conv_wgrad_at(dY, X, layer, idx):
    """dW at flat OIHW indices `idx`."""
    return _sampled(lib().orc_conv_wgrad_at, dY, X, layer, idx)


# ------------------------------------- explicit-im2col GEMM form (full tensors)
#
# The same three convolutions written as the paper's GEMMs on an explicit
# im2col matrix (MicroQonv §II-C, Fig. 2: each receptive field unrolled into a
# column; §IV-A: Y = W_f X', G_W = G_Y X'^T, G_X' = W_f^T G_Y followed by the
# reordering back to the input positions, which sums the copies of one input
# that several receptive fields share).  A library matmul does each fp64
# product; the im2col matrix is built per slice of `nb` batch entries, so the
# full tensors of a large layer fit in host memory.  sum |a*b| (the scale of
# the rounding tolerance) is the same product on |W|, |X'| in fp32.  Slower
# layers are checked with these on the whole output; the 7-loop functions
# above pin them on small layers.

def _im2col(Xn: np.ndarray, layer) -> np.ndarray:
    """X' for a slice of the batch: rows (ci, kh, kw) (the order of W.reshape
    (Cout, -1) for OIHW weights), columns (n, ho, wo).  Zero padding."""
    L = layer
    nb = Xn.shape[0]
    Xp = np.zeros((nb, L.Cin, L.H + 2 * L.pad, L.W + 2 * L.pad), dtype=Xn.dtype)
    Xp[:, :, L.pad:L.pad + L.H, L.pad:L.pad + L.W] = Xn
    cols = np.empty((L.Cin, L.k, L.k, nb, L.Ho, L.Wo), dtype=Xn.dtype)
    for kh in range(L.k):
        for kw in range(L.k):
            win = Xp[:, :, kh:kh + L.stride * (L.Ho - 1) + 1:L.stride, kw:kw + L.stride * (L.Wo - 1) + 1:L.stride]
            cols[:, kh, kw] = win.transpose(1, 0, 2, 3)
    return cols.reshape(L.Cin * L.k * L.k, nb * L.Ho * L.Wo)


def _col2im_add(dXp: np.ndarray, T: np.ndarray, layer) -> None:
    """The reordering of G_X' back to input positions: row (ci, kh, kw),
    column (n, ho, wo) of T adds into padded input (n, ci, ho s + kh,
    wo s + kw)."""
    L = layer
    nb = dXp.shape[0]
    T = T.reshape(L.Cin, L.k, L.k, nb, L.Ho, L.Wo)
    for kh in range(L.k):
        for kw in range(L.k):
            dXp[:, :, kh:kh + L.stride * (L.Ho - 1) + 1:L.stride, kw:kw + L.stride * (L.Wo - 1) + 1:L.stride] += \
                T[:, kh, kw].transpose(1, 0, 2, 3)


def conv_fwd_gemm(X: np.ndarray, W: np.ndarray, layer, nb: int = 8):
    """Y (N, Cout, Ho, Wo) = W_f X' per batch slice, fp64; and sum |a*b| (fp32)."""
    L = layer
    Wf = np.asarray(W, dtype=np.float64).reshape(L.Cout, -1)
    Wa = np.abs(Wf).astype(np.float32)
    Y = np.empty(L.y_shape(), dtype=np.float64)
    Ya = np.empty(L.y_shape(), dtype=np.float64)
    for n0 in range(0, L.N, nb):
        Xc = _im2col(np.asarray(X[n0:n0 + nb], dtype=np.float64), L)
        m = Xc.shape[1] // (L.Ho * L.Wo)
        Y[n0:n0 + m] = (Wf @ Xc).reshape(L.Cout, m, L.Ho, L.Wo).transpose(1, 0, 2, 3)
        Ya[n0:n0 + m] = (Wa @ np.abs(Xc).astype(np.float32)).reshape(L.Cout, m, L.Ho, L.Wo).transpose(1, 0, 2, 3)
    return Y, Ya


def conv_dgrad_gemm(W: np.ndarray, dY: np.ndarray, layer, nb: int = 8):
    """dX (N, Cin, H, W): G_X' = W_f^T G_Y per batch slice, then the
    reordering (col2im sum) into input positions, fp64; and sum |a*b|."""
    L = layer
    Wf = np.asarray(W, dtype=np.float64).reshape(L.Cout, -1)
    Wa = np.abs(Wf).astype(np.float32)
    dX = np.empty(L.x_shape(), dtype=np.float64)
    dXa = np.empty(L.x_shape(), dtype=np.float64)
    P = L.pad
    for n0 in range(0, L.N, nb):
        G = np.asarray(dY[n0:n0 + nb], dtype=np.float64)
        m = G.shape[0]
        Gm = G.transpose(1, 0, 2, 3).reshape(L.Cout, m * L.Ho * L.Wo)
        for out, T in ((dX, Wf.T @ Gm), (dXa, (Wa.T @ np.abs(Gm).astype(np.float32)).astype(np.float64))):
            acc = np.zeros((m, L.Cin, L.H + 2 * P + L.stride, L.W + 2 * P + L.stride), dtype=np.float64)
            _col2im_add(acc, T, L)
            out[n0:n0 + m] = acc[:, :, P:P + L.H, P:P + L.W]
    return dX, dXa


def conv_wgrad_gemm(dY: np.ndarray, X: np.ndarray, layer, nb: int = 8):
    """dW (Cout, Cin, Kh, Kw) = sum over batch slices of G_Y X'^T, fp64; and sum |a*b|."""
    L = layer
    dW = np.zeros((L.Cout, L.Cin * L.k * L.k), dtype=np.float64)
    dWa = np.zeros_like(dW)
    for n0 in range(0, L.N, nb):
        Xc = _im2col(np.asarray(X[n0:n0 + nb], dtype=np.float64), L)
        G = np.asarray(dY[n0:n0 + nb], dtype=np.float64)
        Gm = G.transpose(1, 0, 2, 3).reshape(L.Cout, -1)
        dW += Gm @ Xc.T
        dWa += np.abs(Gm).astype(np.float32) @ np.abs(Xc).astype(np.float32).T
    return dW.reshape(L.w_shape()), dWa.reshape(L.w_shape())


# ------------------------------------------------- instrumented naive flows
#
# These follow MicroQonv §III-C and the Table I comparison: quantization
# applied AFTER im2col.  "Cuyckens et al." extrapolated to convolutions squares
# the im2col-expanded activation matrix X' into 8x8 blocks (and keeps it for
# the backward pass); "DaCapo" re-quantizes X' in line blocks of 64, along
# rows for the forward GEMM and along columns for the backward GEMM.  Each
# flow returns the fake-quantized matrices plus, per original activation
# element, how many quantization events consumed it.

def im2col_index(layer, order: str = "cbf") -> np.ndarray:
    """Index map of X' = im2col(X): shape (Cin*Kh*Kw, Ho*Wo*N), entry = flat
    NCHW index into X, or -1 for a zero-padding position.

    order "cbf": rows (kh, kw, ci), columns (ho, wo, n) -- the channel-batch-
    first X'_{Cin,N} of MicroQonv §IV-A.  order "standard": rows (ci, kh, kw),
    columns (n, ho, wo) -- the usual channel-first im2col of §II-C / Fig. 2,
    on which the naive flows quantize."""
    L = layer
    rows = L.k * L.k * L.Cin
    cols = L.Ho * L.Wo * L.N
    M = np.full((rows, cols), -1, dtype=np.int64)
    n = np.arange(L.N)
    for kh in range(L.k):
        for kw in range(L.k):
            for ci in range(L.Cin):
                r = (kh * L.k + kw) * L.Cin + ci if order == "cbf" else (ci * L.k + kh) * L.k + kw
                for ho in range(L.Ho):
                    hi = ho * L.stride + kh - L.pad
                    if hi < 0 or hi >= L.H:
                        continue
                    for wo in range(L.Wo):
                        wi = wo * L.stride + kw - L.pad
                        if wi < 0 or wi >= L.W:
                            continue
                        if order == "cbf":
                            c = (ho * L.Wo + wo) * L.N + n
                        else:
                            c = (n * L.Ho + ho) * L.Wo + wo
                        M[r, c] = ((n * L.Cin + ci) * L.H + hi) * L.W + wi
    return M


def _fake_quantize_blocks(M: np.ndarray, fmt: str, br: int, bc: int):
    """Two-level microscaling of a 2-D fp64 matrix in br x bc blocks (the same
    steps as the quantizer: tensor scale from the whole matrix, per-block E4M3
    scale, element codes; quotients in fp64 as in mqoracle.c), returning
    fake-quantized values.  A ragged last block row / column is a partial
    block (the same as padding it with zeros, which change no block amax and
    quantize to zero)."""
    M = np.asarray(M, dtype=np.float64)
    grid = format_grid(fmt)
    emax = grid[-1]
    amax = float(np.max(np.abs(M))) if M.size else 0.0
    s_t = tensor_scale(fmt, np.float32(amax))
    R, C = M.shape
    Rp, Cp = -(-R // br) * br, -(-C // bc) * bc
    P = np.zeros((Rp, Cp))
    P[:R, :C] = M
    B = P.reshape(Rp // br, br, Cp // bc, bc)            # block (i, j) is B[i, :, j, :]
    ab = np.abs(B).max(axis=(1, 3))
    bs = decode("e4m3", round_codes("e4m3", ab / (emax * s_t))) if s_t > 0 else np.zeros_like(ab)
    d = (bs * s_t)[:, None, :, None]
    q = np.zeros_like(B)
    np.divide(B, d, out=q, where=np.broadcast_to(d > 0, B.shape))
    out = decode(fmt, round_codes(fmt, q)) * d
    return out.reshape(Rp, Cp)[:R, :C]


def flow_quantize_after_im2col(X: np.ndarray, layer, fmt: str):
    """Cuyckens et al. extrapolated to convolutions: square 8x8 quantization of
    the im2col-expanded X' (quantized once, stored for backward).  Returns
    (X' fake-quantized, index map).  Uses the standard channel-first im2col."""
    idx = im2col_index(layer, "standard")
    Xf = np.asarray(X, dtype=np.float64).ravel()
    M = np.where(idx >= 0, Xf[np.maximum(idx, 0)], 0.0)
    return _fake_quantize_blocks(M, fmt, 8, 8), idx


def flow_dacapo(X: np.ndarray, layer, fmt: str):
    """DaCapo: X' re-quantized in line blocks of 64 -- along K (its columns) for
    the forward GEMM Y = W_f X', along the (Ho Wo N) axis (its rows) for the
    weight-gradient GEMM G_W = G_Y X'^T, on the standard channel-first im2col.
    Returns (fwd X', bwd X', index map)."""
    idx = im2col_index(layer, "standard")
    Xf = np.asarray(X, dtype=np.float64).ravel()
    M = np.where(idx >= 0, Xf[np.maximum(idx, 0)], 0.0)
    return _fake_quantize_blocks(M, fmt, 64, 1), _fake_quantize_blocks(M, fmt, 1, 64), idx


def flow_quantization_counts(layer, flow: str) -> Dict[str, np.ndarray]:
    """Per source element of X, W and G_Y: how many times one training step of
    `flow` quantizes it (Table I's "per elt. quantization").

    Each quantization event is a matrix that gets microscaled, listed with the
    map from its entries to source elements:
      microqonv -- X, W and G_Y each quantized once in square blocks before
                   im2col and reused by all three GEMMs (§IV-A, §IV-B);
      cuyckens  -- the im2col-expanded X' quantized once in squares and stored
                   for backward; W and G_Y once in squares (§III-C);
      dacapo    -- every GEMM operand re-quantized along its own dot-product
                   direction from full precision: X' for the forward and the
                   weight-gradient GEMMs, W_f for the forward and data-gradient
                   GEMMs, G_Y for the data- and weight-gradient GEMMs (§III-C).
    """
    L = layer
    ident = {t: np.arange(n, dtype=np.int64) for t, n in
             (("X", int(np.prod(L.x_shape()))), ("W", int(np.prod(L.w_shape()))),
              ("G", int(np.prod(L.y_shape()))))}
    xprime = im2col_index(L, "standard").ravel()
    events = {
        "microqonv": [("X", ident["X"]), ("W", ident["W"]), ("G", ident["G"])],
        "cuyckens": [("X", xprime), ("W", ident["W"]), ("G", ident["G"])],
        "dacapo": [("X", xprime), ("X", xprime), ("W", ident["W"]), ("W", ident["W"]),
                   ("G", ident["G"]), ("G", ident["G"])],
    }[flow]
    counts = {t: np.zeros(ident[t].size, dtype=np.int64) for t in ident}
    for t, src in events:
        np.add.at(counts[t], src[src >= 0], 1)
    return counts


def backward_storage_bits(layer, flow: str, code_bits: int, scale_bits_per_block: int) -> float:
    """Bits that one flow stores off chip during the forward pass for the
    activation, to bring back in the backward pass (Table I "backward memory
    movement"), per element of X."""
    n_x = int(np.prod(layer.x_shape()))
    packed = code_bits + scale_bits_per_block / 64.0
    if flow == "dacapo":
        return 32.0                                            # full-precision X
    if flow == "cuyckens":
        n_xp = layer.k * layer.k * layer.Cin * layer.Ho * layer.Wo * layer.N
        return packed * n_xp / n_x                             # quantized X' (padding included)
    return packed                                              # quantized X


def gather_im2col_from_packed(q: Dict[str, object], layer):
    """X' gathered from the packed CBF tensor (codes and scales per copy),
    the on-the-fly channel-batch-first im2col of MicroQonv §IV-A.  Returns
    (value matrix, code matrix, scale matrix) with -1 / 0 at padding."""
    idx = im2col_index(layer)
    N, C, H, W = q["dims"]
    flat = idx.copy()
    valid = flat >= 0
    f = np.maximum(flat, 0)
    wi = f % W
    hi = (f // W) % H
    c = (f // (W * H)) % C
    nb = f // (W * H * C)
    blk = ((hi * W + wi) * (N // 8) + nb // 8) * (C // 8) + c // 8
    i = (nb % 8) * 8 + (c % 8)
    codes = unpack_codes(q)
    code_m = np.where(valid, codes[blk, i].astype(np.int64), -1)
    scale_m = np.where(valid, q["scales"][blk], 0)
    vals = dequantize(q).ravel()
    val_m = np.where(valid, vals[f], 0.0)
    return val_m, code_m, scale_m


def unpack_codes(q: Dict[str, object]) -> np.ndarray:
    """Packed code bytes -> (blocks, 64) array of codes (element index i = row*8 + col)."""
    fmt = q["fmt"]
    raw = np.asarray(q["codes"], dtype=np.uint8).reshape(-1, BLOCK_BYTES[fmt])
    if fmt == "e2m1":
        lo = raw & 0xF
        hi = raw >> 4
        return np.stack([lo, hi], axis=-1).reshape(-1, 64)
    if fmt == "e2m3":
        bits = np.unpackbits(raw, axis=1, bitorder="little").reshape(-1, 64, 6)
        return (bits * (1 << np.arange(6, dtype=np.uint8))).sum(axis=2).astype(np.uint8)
    return raw.copy()


# ------------------------------------------------- quantization error (Table II)
#
# MicroQonv §IV-D measures the average per-element quantization MSE of the
# weights (W), activations (A) and output gradients (G), normalized by
# MicroQonv's (Table II: DaCapo 0.891 / 0.982 / 0.827, Cuyckens et al.
# 0.875 / 0.992 / 0.996, MicroQonv+ 0.236 / 1.0 / 1.0 for A / W / G).  The
# pages do not spell the averaging out; the readings taken here:
#   * A is averaged over the valid entries of the standard im2col X' (every
#     copy an operand of the GEMMs; padding excluded) for every flow --
#     MicroQonv's copies all carry their source element's one error;
#   * a flow that quantizes a tensor twice (DaCapo, once per GEMM it feeds)
#     contributes the mean of its two MSEs;
#   * the GEMM matrices are X' (rows (ci, kh, kw), columns (n, ho, wo)),
#     W_f = W.reshape(Cout, Cin Kh Kw) and G_Y as (Cout, N Ho Wo):
#       microqonv  X, W, G quantized once in the CBF 8x8 blocks (§IV-B);
#       cuyckens   8x8 squares of X', W_f and G_Y (§III-C, extrapolated);
#       dacapo     64-line blocks along each GEMM's reduction: X' along K
#                  (fwd) and along (n, ho, wo) (wgrad), W_f along K (fwd) and
#                  along Cout (dgrad), G_Y along Cout (dgrad) and along
#                  (n, ho, wo) (wgrad) (§III-C);
#       microqonv+ as microqonv with the activations in a 6-bit format.

def quantization_mse(X: np.ndarray, W: np.ndarray, G: np.ndarray, layer, fmt: str = "e2m1",
                     fmt_plus: str = "e2m3") -> Dict[str, Dict[str, float]]:
    """Per-element quantization MSE {flow: {"A", "W", "G"}} of one layer's
    tensors (fp32 values; X NCHW, W OIHW, G NCHW) under the flows above."""
    L = layer
    X64, W64, G64 = (np.asarray(a, dtype=np.float64) for a in (X, W, G))
    idx = im2col_index(L, "standard")
    valid = idx >= 0
    Xp = np.where(valid, X64.ravel()[np.maximum(idx, 0)], 0.0)
    Wf = W64.reshape(L.Cout, -1)
    Gm = G64.transpose(1, 0, 2, 3).reshape(L.Cout, -1)

    def mse(Q, R, mask=None):
        e = (Q - R) ** 2
        return float(e[mask].mean() if mask is not None else e.mean())

    def cbf(a, f, role, layout):
        return dequantize(quantize(np.asarray(a, dtype=np.float32), f, role, layout))

    def a_from_x(xhat):      # error of each X' copy = error of its source element
        return mse(np.where(valid, xhat.ravel()[np.maximum(idx, 0)], 0.0), Xp, valid)

    fq = _fake_quantize_blocks
    out = {
        "microqonv": {"A": a_from_x(cbf(X, fmt, "act", "nchw")), "W": mse(cbf(W, fmt, "weight", "oihw"), W64),
                      "G": mse(cbf(G, fmt, "grad", "nchw"), G64)},
        "cuyckens": {"A": mse(fq(Xp, fmt, 8, 8), Xp, valid), "W": mse(fq(Wf, fmt, 8, 8), Wf),
                     "G": mse(fq(Gm, fmt, 8, 8), Gm)},
        "dacapo": {"A": 0.5 * (mse(fq(Xp, fmt, 64, 1), Xp, valid) + mse(fq(Xp, fmt, 1, 64), Xp, valid)),
                   "W": 0.5 * (mse(fq(Wf, fmt, 1, 64), Wf) + mse(fq(Wf, fmt, 64, 1), Wf)),
                   "G": 0.5 * (mse(fq(Gm, fmt, 64, 1), Gm) + mse(fq(Gm, fmt, 1, 64), Gm))},
    }
    out["microqonv+"] = {"A": a_from_x(cbf(X, fmt_plus, "act", "nchw")), "W": out["microqonv"]["W"],
                         "G": out["microqonv"]["G"]}
    return out


def normalized_mse(per_layer, weights=None) -> Dict[str, Dict[str, float]]:
    """Element-weighted mean over layers of each flow's MSE, divided by
    MicroQonv's (Table II's normalization).  weights: {tensor: [count per layer]}."""
    flows, tensors = per_layer[0].keys(), ("A", "W", "G")
    tot = {f: {t: 0.0 for t in tensors} for f in flows}
    for i, m in enumerate(per_layer):
        for f in flows:
            for t in tensors:
                tot[f][t] += m[f][t] * (weights[t][i] if weights else 1.0)
    return {f: {t: tot[f][t] / tot["microqonv"][t] for t in tensors} for f in flows}
