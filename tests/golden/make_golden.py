"""Writes tests/golden/tiny_fp32_oracle.json: the float64 oracle's results on
the tiny fp32 workload (N=64, D=32, C=512, bias, 4 ignored rows, mean,
seed 0), drawn on the CPU.

The source pages print no worked example with numbers, so this fixture is a
regression record of the oracle itself (it calls only ``oracle/`` and the
seeded input generator); the oracle's correctness is pinned separately by
closed forms, finite differences and torch's float64 cross entropy.

Run: python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from linear_cross_entropy_lce_gb300.workloads import make_workload  # noqa: E402
from oracle import lce_oracle as O  # noqa: E402


def tiny_case():
    inp = make_workload("tiny_fp32", device="cpu")
    X = inp["X"].double().numpy()
    W = inp["W"].double().numpy()
    b = inp["b"].double().numpy()
    t = inp["target"].numpy()
    return X, W, b, t


def main():
    X, W, b, t = tiny_case()
    loss, dX, dW, db = O.lce_forward_backward(X, W, b, t, "mean", -100)
    _, lse = O.lce_forward(X, W, b, t, "mean", -100)
    rec = {
        "workload": "tiny_fp32 (N=64, D=32, C=512, bias, 4 ignored, mean, seed 0, CPU generator)",
        "input_checksums": {"X": float(X.sum()), "W": float(W.sum()), "b": float(b.sum()),
                            "target": int(t.sum())},
        "loss": loss,
        "lse_first8": lse[:8].tolist(),
        "dX_row0": dX[0].tolist(),
        "db_first8": db[:8].tolist(),
        "dW_row_target0": dW[int(t[t != -100][0])].tolist(),
        "target0": int(t[t != -100][0]),
        "abs_sums": {"dX": float(np.abs(dX).sum()), "dW": float(np.abs(dW).sum()),
                     "db": float(np.abs(db).sum())},
    }
    with open(os.path.join(HERE, "tiny_fp32_oracle.json"), "w") as f:
        json.dump(rec, f, indent=1)


if __name__ == "__main__":
    main()
