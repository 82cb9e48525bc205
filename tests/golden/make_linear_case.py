"""Writes tests/golden/linear_case.json: a tiny linear-form case for the C ABI
example (tests/c/abi_example.c), every expected value computed by the FP64
oracle (oracle.lce_forward / oracle.lce_backward) from seeded BF16 inputs.

    python tests/golden/make_linear_case.py

The case: N = 6 tokens, H = 16, V = 37 (less than one 256-wide vocabulary
tile, a K range shorter than one 64-wide block), label smoothing 0.1, mean
reduction, one ignored token, targets at both ends of the vocabulary; the
Cut Cross-Entropy card's linear_cross_entropy(embeddings, classifier, labels)
("what_it_does") with the Liger pull request's backward (dX, dW).
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads as wk  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "linear_case.json")


def make():
    n, h, v, eps = 6, 16, 37, 0.1
    x = wk.normal_matrix(21, wk.TID_X, n, h, 1.0, True)  # BF16 bit patterns
    w = wk.normal_matrix(21, wk.TID_W, v, h, h ** -0.5, True)
    y = np.array([3, 36, -100, 0, 17, 5], dtype=np.int64)
    g = [1.0]
    f = oracle.lce_forward(x, w, y, eps, True)
    dx, dw, _ = oracle.lce_backward(x, w, y, f["lse"], f["n_valid"], g, eps, True, z=f["z"])
    return {
        "about": "Written by tests/golden/make_linear_case.py from the FP64 oracle; inputs are "
                 "BF16 bit patterns from the seeded generators in workloads/.",
        "n": n, "h": h, "v": v, "label_smoothing": eps, "reduce_loss": 1, "ignore_idx": -100,
        "grad_output": g, "target": y.tolist(),
        "x_bf16_bits": x.ravel().astype(int).tolist(), "w_bf16_bits": w.ravel().astype(int).tolist(),
        "loss": float(f["loss"]), "n_valid": int(f["n_valid"]), "lse": f["lse"].tolist(),
        "dX": dx.ravel().tolist(), "dW": dw.ravel().tolist(),
    }


if __name__ == "__main__":
    with open(OUT, "w") as fh:
        json.dump(make(), fh, indent=1)
        fh.write("\n")
    print(OUT)
