"""Pins for the oracle's direct 7-loop fp64 convolutions.

Independent checks: torch's fp64 CPU conv2d / conv2d_input / conv2d_weight
(library routines), the paper's own GEMM formulation over an explicitly built
im2col matrix (MicroQonv §II-C and §IV-A: Y = W_f X', G_W = G_Y X'^T,
G_X' = W_f^T G_Y followed by the col2im sum), the adjoint identity
<fwd(X), dY> = <X, dgrad(dY)>, and the 1x1 stride-1 case reducing to a matmul.
"""
import numpy as np
import pytest
import torch

from synthetic import Layer

GEOMS = [
    Layer(8, 16, 8, 8, 16, 3, 1, 1),
    Layer(8, 8, 7, 5, 16, 3, 2, 1),
    Layer(8, 16, 6, 6, 8, 1, 2, 0),
    Layer(16, 8, 5, 9, 8, 3, 1, 0),
    Layer(8, 8, 9, 9, 8, 5, 2, 2),
    Layer(8, 8, 4, 4, 8, 1, 1, 0),
]


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("L", GEOMS, ids=lambda L: L.name())
def test_conv_matches_torch_fp64(orc, L):
    X, W, dY = rand(L.x_shape(), 1), rand(L.w_shape(), 2), rand(L.y_shape(), 3)
    Xt, Wt, dYt = (torch.from_numpy(a) for a in (X, W, dY))
    Y, Ya = orc.conv_fwd(X, W, L)
    ref = torch.nn.functional.conv2d(Xt, Wt, stride=L.stride, padding=L.pad).numpy()
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)
    refa = torch.nn.functional.conv2d(Xt.abs(), Wt.abs(), stride=L.stride, padding=L.pad).numpy()
    np.testing.assert_allclose(Ya, refa, rtol=1e-12, atol=1e-12)

    dX, dXa = orc.conv_dgrad(W, dY, L)
    ref = torch.nn.grad.conv2d_input(Xt.shape, Wt, dYt, stride=L.stride, padding=L.pad).numpy()
    np.testing.assert_allclose(dX, ref, rtol=1e-12, atol=1e-12)
    refa = torch.nn.grad.conv2d_input(Xt.shape, Wt.abs(), dYt.abs(), stride=L.stride, padding=L.pad).numpy()
    np.testing.assert_allclose(dXa, refa, rtol=1e-12, atol=1e-12)

    dW, dWa = orc.conv_wgrad(dY, X, L)
    ref = torch.nn.grad.conv2d_weight(Xt, Wt.shape, dYt, stride=L.stride, padding=L.pad).numpy()
    np.testing.assert_allclose(dW, ref, rtol=1e-12, atol=1e-12)
    refa = torch.nn.grad.conv2d_weight(Xt.abs(), Wt.shape, dYt.abs(), stride=L.stride, padding=L.pad).numpy()
    np.testing.assert_allclose(dWa, refa, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L", GEOMS[:5], ids=lambda L: L.name())
def test_conv_matches_paper_gemm_forms(orc, L):
    """The three GEMMs of MicroQonv §IV-A on the channel-batch-first im2col X'."""
    X, W, dY = rand(L.x_shape(), 4), rand(L.w_shape(), 5), rand(L.y_shape(), 6)
    idx = orc.im2col_index(L)                                   # (Kh Kw Cin) x (Ho Wo N)
    Xp = np.where(idx >= 0, X.ravel()[np.maximum(idx, 0)], 0.0)
    Wf = W.transpose(0, 2, 3, 1).reshape(L.Cout, -1)            # rows co, cols (kh, kw, ci)
    Gy = dY.transpose(1, 2, 3, 0).reshape(L.Cout, -1)           # rows co, cols (ho, wo, n)
    # forward: Y = W_f X'
    Y = (Wf @ Xp).reshape(L.Cout, L.Ho, L.Wo, L.N).transpose(3, 0, 1, 2)
    np.testing.assert_allclose(orc.conv_fwd(X, W, L)[0], Y, rtol=1e-12, atol=1e-12)
    # weight gradient: G_W = G_Y X'^T
    Gw = (Gy @ Xp.T).reshape(L.Cout, L.k, L.k, L.Cin).transpose(0, 3, 1, 2)
    np.testing.assert_allclose(orc.conv_wgrad(dY, X, L)[0], Gw, rtol=1e-12, atol=1e-12)
    # data gradient: G_X' = W_f^T G_Y, then col2im sums every copy into its source pixel
    Gxp = Wf.T @ Gy
    dX = np.zeros(X.size)
    np.add.at(dX, idx[idx >= 0], Gxp[idx >= 0])
    np.testing.assert_allclose(orc.conv_dgrad(W, dY, L)[0], dX.reshape(X.shape), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("L", GEOMS, ids=lambda L: L.name())
def test_dgrad_is_adjoint_of_fwd(orc, L):
    X, W, dY = rand(L.x_shape(), 7), rand(L.w_shape(), 8), rand(L.y_shape(), 9)
    lhs = np.sum(orc.conv_fwd(X, W, L)[0] * dY)
    rhs = np.sum(X * orc.conv_dgrad(W, dY, L)[0])
    wg = np.sum(W * orc.conv_wgrad(dY, X, L)[0])
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))
    assert abs(lhs - wg) <= 1e-10 * max(1.0, abs(lhs))


def test_1x1_is_matmul(orc):
    L = Layer(8, 16, 3, 4, 24, 1, 1, 0)
    X, W = rand(L.x_shape(), 10), rand(L.w_shape(), 11)
    Y = np.einsum("oc,nchw->nohw", W[:, :, 0, 0], X)
    np.testing.assert_allclose(orc.conv_fwd(X, W, L)[0], Y, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("L", GEOMS[:3], ids=lambda L: L.name())
def test_sampled_equals_full(orc, L):
    X, W, dY = rand(L.x_shape(), 12), rand(L.w_shape(), 13), rand(L.y_shape(), 14)
    rng = np.random.default_rng(0)
    for full, at, A, B, shp in (
        (orc.conv_fwd, orc.conv_fwd_at, X, W, L.y_shape()),
        (orc.conv_dgrad, orc.conv_dgrad_at, W, dY, L.x_shape()),
        (orc.conv_wgrad, orc.conv_wgrad_at, dY, X, L.w_shape()),
    ):
        ref, refa = full(A, B, L)
        idx = rng.integers(0, int(np.prod(shp)), 50)
        v, va = at(A, B, L, idx)
        np.testing.assert_array_equal(v, ref.ravel()[idx])
        np.testing.assert_array_equal(va, refa.ravel()[idx])


@pytest.mark.parametrize("nb", [8, 3])
@pytest.mark.parametrize("L", GEOMS + [Layer(16, 24, 7, 6, 16, 3, 2, 2), Layer(8, 16, 11, 12, 16, 5, 2, 2)],
                         ids=lambda L: L.name() if hasattr(L, "name") else str(L))
def test_explicit_im2col_gemm_checker_matches_7_loop(orc, L, nb):
    """The full-tensor checker (explicit im2col + library fp64 matmul, batch
    slices of nb entries, the last one ragged for nb = 3) equals the direct
    7-loop oracle; its sum |a*b|, formed in fp32, is within fp32 rounding."""
    X, W, dY = rand(L.x_shape(), 21), rand(L.w_shape(), 22), rand(L.y_shape(), 23)
    for gemm, loop, A, B in ((orc.conv_fwd_gemm, orc.conv_fwd, X, W), (orc.conv_dgrad_gemm, orc.conv_dgrad, W, dY),
                             (orc.conv_wgrad_gemm, orc.conv_wgrad, dY, X)):
        v, va = gemm(A, B, L, nb=nb)
        ref, refa = loop(A, B, L)
        np.testing.assert_allclose(v, ref, rtol=1e-11, atol=1e-11 * np.abs(ref).max())
        np.testing.assert_allclose(va, refa, rtol=1e-5, atol=1e-6 * refa.max())
