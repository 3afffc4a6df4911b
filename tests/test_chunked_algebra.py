"""The chunked evaluation the GPU paths implement, checked in fp64 on the CPU.

Both CUDA paths evaluate the recurrence in 64-token chunks with a WY/UT form of the
products of the transitions alpha_t (I - beta_t k_t k_t^T) (notes on PRISM, section
2.2) and pass the state between chunks with the associative combine of input-only
affine maps S -> S M + N (notes, section 2.1).  This file restates those steps in
numpy, exactly as the tensor-core kernel arranges them (decay factors relative to
the chunk end, the augmented segment map Z = [N; M], the per-chunk (o0, Qhat) stash,
the segment combine and the fix-up), and checks the result against the sequential
oracle on the same inputs.  A mismatch on the GPU with this test green points at the
kernels' data movement, not at the algebra.
"""
import numpy as np
import pytest
import scipy.special as sps

from ssm_sequence_layer_gb300.inputs import make_inputs

C = 64


def prep(v, w, gamma, eta):
    """x_{t,l} = gamma_{t,l} g_t r_{t,l} for one sequence; v [T,dv], w [4,dv]."""
    T, dv = v.shape
    h = np.zeros_like(v)
    for j in range(4):
        h[j:] += w[j] * v[: T - j]
    Phi = sps.ndtr(h)
    g = Phi + h * np.exp(-h * h / 2) / np.sqrt(2 * np.pi)
    r = v - h * Phi
    R = gamma.shape[1]
    X = np.zeros((T, R, dv))
    for l in range(R):
        X[:, l] = gamma[:, l, None] * g * r
        r = r * (1 - eta[:, l, None] * g)
    return X


def chunk_maps(q, k, v, beta, alpha, u, X):
    """Per chunk: the factors the kernel builds.  Returns a list of dicts."""
    T, dk = q.shape
    out = []
    for t0 in range(0, T, C):
        n = min(C, T - t0)
        pad = lambda a: np.concatenate([a[t0:t0 + n], np.zeros((C - n,) + a.shape[1:])]) if n < C else a[t0:t0 + C]
        Q, K, V, Uc, Xc = pad(q), pad(k), pad(v), pad(u), pad(X)
        b = np.concatenate([beta[t0:t0 + n], np.zeros(C - n)])
        la = np.concatenate([np.log(alpha[t0:t0 + n]), np.zeros(C - n)])
        lam = np.cumsum(la)
        lc = lam[-1]
        rowf, colf = np.exp(lam - lc), np.exp(lc - lam)
        Gam = np.exp(lam)
        strict = np.tril(np.ones((C, C)), -1)
        incl = np.tril(np.ones((C, C)))
        A = (b[:, None] * np.exp(lam[:, None] - lam[None, :]) * (K @ K.T)) * strict
        Tm = np.linalg.inv(np.eye(C) + A)
        R = Uc.shape[1]
        Xs = Xc * colf[:, None, None]
        MX = np.zeros((C, V.shape[1]))
        for l in range(R):
            PK = (b[:, None] * rowf[:, None] * (K @ Uc[:, l].T)) * strict
            MX += PK @ Xs[:, l]
        RHS = b[:, None] * V - MX
        Up = Tm @ RHS
        W = Tm @ (b[:, None] * Gam[:, None] * K)
        UWs = np.concatenate([Up.T, W.T]) * colf[None, :]             # [U'^T; W^T] diag(colf)
        G = (rowf[:, None] * (Q @ K.T)) * incl
        D4 = UWs @ G.T
        D5 = UWs @ K
        for l in range(R):
            PQ = (rowf[:, None] * (Q @ Uc[:, l].T)) * incl
            XsT0 = np.concatenate([Xs[:, l].T, np.zeros_like(Xs[:, l].T)])  # [Xs^T; 0]
            D4 += XsT0 @ PQ.T
            D5 += XsT0 @ Uc[:, l]
        dvv = V.shape[1]
        Oloc_T, GW_T = D4[:dvv], D4[dvv:]
        Nc, WtK = D5[:dvv], D5[dvv:]
        Qt = Gam[None, :] * Q.T - GW_T
        Mc = np.exp(lc) * np.eye(dk) - WtK
        out.append(dict(n=n, Qt=Qt, Mc=Mc, Nc=Nc, Oloc_T=Oloc_T))
    return out


def chunked_forward(q, k, v, beta, alpha, u, X, P):
    T, dk = q.shape
    dv = v.shape[1]
    ch = chunk_maps(q, k, v, beta, alpha, u, X)
    NC = len(ch)
    out = np.zeros((T, dv))
    zsum, stash = [], {}
    for p in range(P):
        cb, ce = p * NC // P, (p + 1) * NC // P
        Z = np.zeros((dv + dk, dk))
        if p > 0:
            Z[dv:] = np.eye(dk)
        for c in range(cb, ce):
            m = ch[c]
            D7 = Z @ m["Qt"]                                   # [N Qt; M Qt]
            o0 = (D7[:dv] + m["Oloc_T"]).T                     # token-major
            Qhat = D7[dv:].T
            if p == 0:
                out[c * C: c * C + m["n"]] = o0[: m["n"]]
            else:
                stash[c] = (o0, Qhat)
            Z = Z @ m["Mc"] + np.concatenate([m["Nc"], np.zeros((dk, dk))])
        zsum.append(Z)
    S = np.zeros((dv, dk))
    starts = [S]
    for p in range(1, P):
        S = S @ zsum[p - 1][dv:] + zsum[p - 1][:dv]
        starts.append(S)
    for p in range(1, P):
        cb, ce = p * NC // P, (p + 1) * NC // P
        for c in range(cb, ce):
            o0, Qhat = stash[c]
            n = ch[c]["n"]
            out[c * C: c * C + n] = (o0 + Qhat @ starts[p].T)[:n]
    return out


@pytest.mark.parametrize("T,L,P", [(64, 1, 1), (200, 3, 1), (200, 3, 3), (513, 4, 5), (700, 2, 11)])
def test_chunked_algebra_matches_oracle(oracle_mod, T, L, P):
    inp = make_inputs(1, 1, T, 64, 64, L, dtype="f32", seed=40 + T + P)
    a = {k: (v.double().numpy()[0, 0] if hasattr(v, "double") and k != "conv_w" else v) for k, v in inp.items()}
    w = inp["conv_w"].double().numpy()[0]
    R = L - 1
    X = prep(a["v"], w, a["gamma"], a["eta"]) if R > 0 else np.zeros((T, 0, 64))
    u = a["u"] if R > 0 else np.zeros((T, 0, 64))
    got = chunked_forward(a["q"], a["k"], a["v"], a["beta"], a["alpha"], u, X, P)
    ref = oracle_mod.forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"], inp["gamma"],
                             inp["eta"], inp["conv_w"], L)["out"][0, 0]
    err = np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2))
    assert err < 1e-10, err
