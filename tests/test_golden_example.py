"""The worked example in tests/golden (dk = dv = 2, L = 3, six tokens).

The fixture's expected values were written by tests/golden/make_golden.py from the
oracle, so comparing the oracle to them only guards against regressions.  The pin
is the second test: the first two tokens re-derived by hand in 50-digit mpmath
from the definition (anchor, exact-erf GELU gain and residual, residual chain,
GDN transition, rank-L write, readout of the post-update state).
"""
import json
import os

import mpmath as mp
import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load():
    with open(os.path.join(HERE, "golden", "worked_example_T6.json")) as f:
        return json.load(f)


def test_oracle_reproduces_worked_example(oracle_mod):
    ex = load()
    a = {n: np.array(ex[n], dtype=np.float64)[None, None] for n in
         ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")}
    res = oracle_mod.forward(a["q"], a["k"], a["v"], a["beta"], a["alpha"], a["u"], a["gamma"],
                             a["eta"], np.array(ex["conv_w"]), ex["L"], want_state=True)
    np.testing.assert_allclose(res["out"][0, 0], np.array(ex["expected"]["out"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(res["S_final"][0, 0], np.array(ex["expected"]["S_final"]), rtol=0, atol=1e-15)


def test_first_two_tokens_by_hand():
    mp.mp.dps = 50
    ex = load()
    w = ex["conv_w"][0]
    v, k, q, u = ex["v"], ex["k"], ex["q"], ex["u"]
    dk = dv = 2

    def mpv(x):
        return [mp.mpf(repr(float(z))) for z in x]

    def Phi(x):
        return (1 + mp.erf(x / mp.sqrt(2))) / 2

    def phi(x):
        return mp.exp(-x * x / 2) / mp.sqrt(2 * mp.pi)

    S = [[mp.mpf(0)] * dk for _ in range(dv)]
    outs = []
    for t in range(2):
        h = [sum(mp.mpf(repr(w[j][c])) * mp.mpf(repr(v[t - j][c])) for j in range(4) if t - j >= 0)
             for c in range(dv)]
        g = [Phi(x) + x * phi(x) for x in h]
        e = [mp.mpf(repr(v[t][c])) - h[c] * Phi(h[c]) for c in range(dv)]
        al, be = mp.mpf(repr(ex["alpha"][t])), mp.mpf(repr(ex["beta"][t]))
        kt, vt, qt = mpv(k[t]), mpv(v[t]), mpv(q[t])
        Sk = [sum(S[i][j] * kt[j] for j in range(dk)) for i in range(dv)]
        S = [[al * (S[i][j] - be * Sk[i] * kt[j]) + be * vt[i] * kt[j] for j in range(dk)] for i in range(dv)]
        r = e[:]
        for l in range(2):
            gm = mp.mpf(repr(ex["gamma"][t][l]))
            ul = mpv(u[t][l])
            for i in range(dv):
                for j in range(dk):
                    S[i][j] += gm * g[i] * r[i] * ul[j]
            et = mp.mpf(repr(ex["eta"][t][l]))
            r = [r[i] * (1 - et * g[i]) for i in range(dv)]
        outs.append([float(sum(S[i][j] * qt[j] for j in range(dk))) for i in range(dv)])
    np.testing.assert_allclose(np.array(outs), np.array(ex["expected"]["out"][:2]), rtol=1e-14, atol=1e-15)
