"""Write tests/golden/worked_example_T6.json: a hand-sized worked example of the
PRISM recurrence (dk = dv = 2, L = 3, six tokens, round-number inputs) with the
outputs of the fp64 oracle.  Calls only oracle/.  Re-run after a change of the
oracle's arithmetic that a passage of the pages justifies, and name that passage
in the commit.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import prism_oracle  # noqa: E402


def example():
    T, dk, dv, L = 6, 2, 2, 3
    q = [[1.0, 0.0], [0.6, 0.8], [0.0, 1.0], [0.8, -0.6], [-1.0, 0.0], [0.6, 0.8]]
    k = [[1.0, 0.0], [0.0, 1.0], [0.6, 0.8], [0.8, 0.6], [0.0, -1.0], [-0.6, 0.8]]
    v = [[1.0, -0.5], [0.25, 2.0], [-1.5, 0.5], [0.0, 1.0], [2.0, -2.0], [0.5, 0.5]]
    beta = [0.5, 0.25, 0.75, 1.0, 0.5, 0.125]
    alpha = [0.9, 0.8, 1.0, 0.5, 0.75, 0.95]
    u = [[[0.0, 1.0], [1.0, 0.0]], [[0.6, 0.8], [0.8, -0.6]], [[1.0, 0.0], [0.0, 1.0]],
         [[-0.8, 0.6], [0.6, 0.8]], [[0.0, -1.0], [1.0, 0.0]], [[0.8, 0.6], [-0.6, 0.8]]]
    gamma = [[0.5, 0.25], [0.75, 0.5], [0.25, 0.25], [1.0, 0.5], [0.5, 0.75], [0.125, 0.5]]
    eta = [[0.5, 0.0], [0.25, 0.0], [0.75, 0.0], [1.0, 0.0], [0.5, 0.0], [0.125, 0.0]]
    conv_w = [[[0.5, -0.25], [0.25, 0.5], [-0.5, 0.25], [0.125, 0.0]]]
    return dict(T=T, dk=dk, dv=dv, L=L, q=q, k=k, v=v, beta=beta, alpha=alpha, u=u,
                gamma=gamma, eta=eta, conv_w=conv_w)


def main():
    ex = example()
    a = {n: np.array(ex[n], dtype=np.float64)[None, None] for n in
         ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")}
    w = np.array(ex["conv_w"], dtype=np.float64)
    res = prism_oracle.forward(a["q"], a["k"], a["v"], a["beta"], a["alpha"], a["u"], a["gamma"],
                               a["eta"], w, ex["L"], want_state=True, want_hge=True, want_x=True)
    ex["expected"] = {
        "out": res["out"][0, 0].tolist(), "S_final": res["S_final"][0, 0].tolist(),
        "h": res["h"][0, 0].tolist(), "g": res["g"][0, 0].tolist(), "e": res["e"][0, 0].tolist(),
        "X": res["X"][0, 0].tolist(),
    }
    ex["source"] = "outputs written by tests/golden/make_golden.py from the fp64 oracle"
    with open(os.path.join(HERE, "worked_example_T6.json"), "w") as f:
        json.dump(ex, f, indent=1)


if __name__ == "__main__":
    main()
