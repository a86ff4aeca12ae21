"""Table II's normalized per-element quantization MSE (MicroQonv §IV-D) on the
synthetic ResNet-32 / CIFAR-shaped layers (the pages' network, with seeded
synthetic tensors standing in for its trained ones), from the oracle alone.

    python -m oracle.mse_report [--json]

Prints, per layer and element-weighted over the five layers, each flow's MSE
of A, W and G divided by MicroQonv's, next to the values Table II prints, and
whether the orderings the paper reads from them hold here.
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import synthetic as S  # noqa: E402

PRINTED = {"dacapo": (0.891, 0.982, 0.827), "cuyckens": (0.875, 0.992, 0.996),
           "microqonv": (1.0, 1.0, 1.0), "microqonv+": (0.236, 1.0, 1.0)}


def measure(wl=S.WORKLOADS[1]):
    per_layer, counts = [], {"A": [], "W": [], "G": []}
    for li, L in enumerate(wl.layers):
        X, W, G = S.draw_x(wl, li), S.draw_w(wl, li), S.draw_dy(wl, li)
        per_layer.append(oracle.quantization_mse(X, W, G, L, wl.fmt))
        counts["A"].append(int((oracle.im2col_index(L, "standard") >= 0).sum()))
        counts["W"].append(W.size)
        counts["G"].append(G.size)
    return per_layer, oracle.normalized_mse(per_layer, counts)


def main():
    per_layer, norm = measure()
    ordering = {
        "activation MSE higher for MicroQonv than the im2col flows":
            norm["cuyckens"]["A"] < 1.0 and norm["dacapo"]["A"] < 1.0,
        "line-block (DaCapo) gradient MSE below the square-block ones":
            norm["dacapo"]["G"] < min(1.0, norm["cuyckens"]["G"]),
        "weight MSE alike across flows (within 5%)":
            all(abs(norm[f]["W"] - 1.0) < 0.05 for f in norm),
        "6-bit activations cut the activation MSE": norm["microqonv+"]["A"] < 0.5,
    }
    if "--json" in sys.argv:
        print(json.dumps({"normalized": norm, "printed": PRINTED, "ordering_holds": ordering}))
        return
    print("flow          A (here / Table II)   W (here / Table II)   G (here / Table II)")
    for f in ("dacapo", "cuyckens", "microqonv", "microqonv+"):
        print(f"{f:<12}" + "".join(f"   {norm[f][t]:.3f} / {PRINTED[f][i]:.3f}     "
                                   for i, t in enumerate(("A", "W", "G"))))
    for k, v in ordering.items():
        print(f"{'holds' if v else 'does not hold'}: {k}")


if __name__ == "__main__":
    main()
