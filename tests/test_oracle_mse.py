"""Pins for the oracle's per-element quantization MSE (MicroQonv §IV-D,
Table II) and a regression check of the orderings it reports.

  * closed form: 8x8 weight blocks holding one maxB_ef * 448 * 2^j element
    and 63 copies of 0.75 * 448 * 2^j (a rounding midpoint of E2M1, which
    goes to the even code 1.0) have per-element error 0.25 * 448 * 2^j on
    63 of 64 elements; for a 1x1 layer the 8x8 squares of W_f are the
    MicroQonv blocks, so both flows give exactly that;
  * the activation error averaged over X' copies equals the per-element
    error of X weighted by each element's im2col copy count (counted by the
    independent instrumented flow);
  * scaling every tensor by a power of two scales every MSE by its square,
    exactly, and leaves the normalized table unchanged.
"""
import numpy as np
import pytest

import synthetic as S
from synthetic import Layer


def test_closed_form_weight_mse(orc):
    L = Layer(8, 16, 4, 4, 16, 1, 1, 0)
    j = -5
    W = np.full(L.w_shape(), 0.75 * 448 * 2.0 ** j, dtype=np.float32)
    W[::8, ::8] = 6.0 * 448 * 2.0 ** j                 # one maximum per 8x8 block
    X = np.full(L.x_shape(), 6.0 * 448 * 2.0 ** -3, dtype=np.float32)    # T_scale 2^-3: exact
    G = np.full(L.y_shape(), 6.0 * 448 * 2.0 ** -9, dtype=np.float32)
    m = orc.quantization_mse(X, W, G, L, "e2m1")
    expect = 63 / 64 * (0.25 * 448 * 2.0 ** j) ** 2
    assert m["microqonv"]["W"] == pytest.approx(expect, rel=1e-12)
    assert m["cuyckens"]["W"] == pytest.approx(expect, rel=1e-12)
    assert m["microqonv"]["A"] == 0.0 and m["microqonv"]["G"] == 0.0   # constants on the grid: exact


def test_activation_error_weighted_by_im2col_copies(orc):
    L = Layer(8, 16, 6, 5, 8, 3, 1, 1)
    wl = S.WORKLOADS[0]
    X = S.draw_x(wl, 0, L.x_shape())
    W = S.draw_w(wl, 0, L.w_shape())
    G = S.draw_dy(wl, 0, L.y_shape())
    m = orc.quantization_mse(X, W, G, L, "e2m1")
    xhat = orc.dequantize(orc.quantize(X, "e2m1", "act", "nchw"))
    count = orc.flow_quantization_counts(L, "cuyckens")["X"]      # copies of each element in X'
    e2 = ((xhat - X.astype(np.float64)) ** 2).ravel()
    assert m["microqonv"]["A"] == pytest.approx(float((count * e2).sum() / count.sum()), rel=1e-12)


def test_power_of_two_scaling(orc):
    L = Layer(8, 16, 6, 6, 16, 3, 1, 1)
    wl = S.WORKLOADS[1]
    X, W, G = S.draw_x(wl, 0, L.x_shape()), S.draw_w(wl, 0, L.w_shape()), S.draw_dy(wl, 0, L.y_shape())
    a = orc.quantization_mse(X, W, G, L)
    b = orc.quantization_mse(X * np.float32(0.125), W * np.float32(0.125), G * np.float32(0.125), L)
    for f in a:
        for t in "AWG":
            assert b[f][t] == a[f][t] / 64.0
    assert orc.normalized_mse([a]) == orc.normalized_mse([b])


@pytest.mark.slow
def test_table2_orderings_on_resnet32_layers():
    """The orderings the paper reads from Table II, on the synthetic
    ResNet-32-shaped layers (oracle.mse_report)."""
    from oracle import mse_report
    _, norm = mse_report.measure()
    assert norm["cuyckens"]["A"] < 1.0 and norm["dacapo"]["A"] < 1.0
    assert norm["dacapo"]["G"] < min(1.0, norm["cuyckens"]["G"])
    assert norm["microqonv+"]["A"] < 0.5
