"""Writes streamkl_small.json: fixed small inputs and their expected outputs.

Case "dyadic": values on a 1/4 grid in [-2, 2] (exact in bf16), B = 1,
H = 2, NQ = NK = 6, d1 = 4, d2 = 2, causal, s1 = 0.5, s2 = 0.75; expected
KL, LSE1, LSE2 and the gradients of both modes (dKL = 1) from the float64
oracle (the pages print no worked example to take them from).

Case "bernoulli": one query row, two keys, d = 2, s = 1, student logits
zero: P1 = (p, 1 - p) with p = e / (e + 1), P2 = (1/2, 1/2), so
KL = p log(2p) + (1 - p) log(2(1 - p)), LSE1 = log(e + 1), LSE2 = log 2
(the definition of the row-wise KL between the two attention rows, StreamKL
article, "Why attention distillation matters"), written here with ``math``.

Run from the repository root: python tests/golden/make_golden.py
"""

import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def dyadic(shape, a, b, c):
    """Deterministic values on the 1/4 grid in [-2, 2]."""
    out = np.empty(shape)
    for idx in np.ndindex(*shape):
        h, i, j = idx[-3], idx[-2], idx[-1]
        out[idx] = ((a * i + b * j + c * h) % 17 - 8) / 4.0
    return out


def main():
    q1 = dyadic((1, 2, 6, 4), 3, 5, 7)
    k1 = dyadic((1, 2, 6, 4), 5, 2, 3)
    q2 = dyadic((1, 2, 6, 2), 7, 3, 1)
    k2 = dyadic((1, 2, 6, 2), 2, 7, 5)
    s1, s2 = 0.5, 0.75
    kl, l1, l2 = oracle.forward(q1, k1, q2, k2, s1, True, scale2=s2)
    dkl = np.ones((1, 2, 6))
    g2 = oracle.backward(q1, k1, q2, k2, s1, True, dkl, oracle.MODE_P2, scale2=s2)
    g1 = oracle.backward(q1, k1, q2, k2, s1, True, dkl, oracle.MODE_P1, scale2=s2)
    p = math.e / (math.e + 1.0)
    cases = {
        "dyadic": {
            "expected_from": "float64 oracle (oracle.forward / oracle.backward)",
            "causal": True, "scale1": s1, "scale2": s2,
            "q1": q1.tolist(), "k1": k1.tolist(), "q2": q2.tolist(), "k2": k2.tolist(),
            "kl": kl.tolist(), "lse1": l1.tolist(), "lse2": l2.tolist(),
            "dq2_p2": g2[0].tolist(), "dk2_p2": g2[1].tolist(),
            "dq1_p1": g1[0].tolist(), "dk1_p1": g1[1].tolist(),
        },
        "bernoulli": {
            "expected_from": "closed form: p = e/(e+1), KL = p log 2p + (1-p) log 2(1-p)",
            "causal": False, "scale1": 1.0, "scale2": 1.0,
            "q1": [[[[1.0, 0.0]]]], "k1": [[[[1.0, 0.0], [0.0, 0.0]]]],
            "q2": [[[[0.0, 0.0]]]], "k2": [[[[1.0, 0.0], [0.0, 1.0]]]],
            "kl": [[[p * math.log(2 * p) + (1 - p) * math.log(2 * (1 - p))]]],
            "lse1": [[[math.log(math.e + 1.0)]]], "lse2": [[[math.log(2.0)]]],
        },
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "streamkl_small.json")
    with open(path, "w") as f:
        json.dump(cases, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
