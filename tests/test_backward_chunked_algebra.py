"""The chunk-parallel arrangement of the backward pass, checked in fp64 on the CPU.

The backward's two sequential passes (the states S_{t-1} forward, the state cotangents dS_t
in reverse) can run chunk by chunk, every chunk at once, once the value of each at the chunk
boundaries is known:
  * the states entering each chunk are what the forward's chunked evaluation already forms
    (the state passed between chunks, notes on PRISM, section 2.1);
  * the cotangent carry dS_t = dS_{t+1} A_{t+1} + dout_t q_t^T, with A = alpha (I - beta k k^T)
    symmetric, is itself a recurrence of the forward's family run backwards in time: with
    s = T - 1 - t it reads G_s = G_{s-1} A'_s + x'_s u'_s^T, where step s takes the gates and
    key of token T - s (one token later than the write's token T - 1 - s), the write is rank 1
    with u' = q and x' = dout of token T - 1 - s, the GDN write is absent (v' = 0), step 0 has
    the identity transition (alpha' = 1, beta' = 0) and the initial value is dS_final.
This file restates that mapping in numpy and checks (1) the reversed recurrence reproduces the
sequential cotangents token by token and (2) per-chunk backward passes started from those
boundary values, followed by the token-local chain and convolution backwards, give every
cotangent of the fp64 backward oracle.
"""
import numpy as np
import pytest

from oracle import prism_backward
from ssm_sequence_layer_gb300.inputs import make_cotangents, make_inputs

C = 64


def forward_family(alpha, beta, k, v, x, u, S0):
    """S_s = alpha_s S_{s-1} (I - beta_s k_s k_s^T) + beta_s v_s k_s^T + sum_l x_{s,l} u_{s,l}^T,
    every state returned ([T+1] states, index s+1 holds S_s, index 0 holds S0)."""
    T = len(alpha)
    out = [S0]
    S = S0
    for s in range(T):
        y = S @ k[s]
        S = alpha[s] * (S - beta[s] * np.outer(y, k[s])) + beta[s] * np.outer(v[s], k[s])
        for l in range(u.shape[1]):
            S = S + np.outer(x[s, l], u[s, l])
        out.append(S)
    return out


def factors(v, w, gamma, eta):
    """x_{t,l} = gamma g r_l, with g, r from the anchor (one sequence; v [T,dv], w [4,dv])."""
    from scipy.special import ndtr
    T, dv = v.shape
    h = np.zeros_like(v)
    for j in range(4):
        h[j:] += w[j] * v[: T - j]
    Phi = ndtr(h)
    g = Phi + h * np.exp(-h * h / 2) / np.sqrt(2 * np.pi)
    r = v - h * Phi
    X = np.zeros((T, gamma.shape[1], dv))
    for l in range(gamma.shape[1]):
        X[:, l] = gamma[:, l, None] * g * r
        r = r * (1 - eta[:, l, None] * g)
    return X


def case(T=200, dk=16, dv=12, L=3, seed=2):
    inp = make_inputs(1, 1, T, dk, dv, L, dtype="f32", seed=seed)
    x = {n: inp[n].double().numpy()[0, 0] for n in ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")}
    x["conv_w"] = inp["conv_w"].double().numpy()[0]
    dout, dS_final = make_cotangents(1, 1, T, dk, dv, seed=seed, with_state=True)
    return inp, x, dout.double().numpy()[0, 0], dS_final.double().numpy()[0, 0]


def adjoint_sequential(x, dout, dS_final):
    """dS_t (cotangent of S_t, readout of token t included) for every t, token by token."""
    T = len(x["alpha"])
    G = [None] * T
    cur = dS_final + np.outer(dout[T - 1], x["q"][T - 1])
    G[T - 1] = cur
    for t in range(T - 2, -1, -1):
        kk = x["k"][t + 1]
        cur = x["alpha"][t + 1] * (cur - x["beta"][t + 1] * np.outer(cur @ kk, kk)) + np.outer(dout[t], x["q"][t])
        G[t] = cur
    return G


def adjoint_as_forward(x, dout, dS_final):
    """The same cotangents from the forward family on the reversed, shifted sequence."""
    T = len(x["alpha"])
    dk, dv = x["q"].shape[1], dout.shape[1]
    idx_w = np.arange(T - 1, -1, -1)                      # write of step s: token T - 1 - s
    idx_a = np.concatenate([[0], np.arange(T - 1, 0, -1)])  # transition of step s >= 1: token T - s
    alpha = np.where(np.arange(T) == 0, 1.0, x["alpha"][idx_a])
    beta = np.where(np.arange(T) == 0, 0.0, x["beta"][idx_a])
    k = x["k"][idx_a]
    v = np.zeros((T, dv))
    xs = dout[idx_w][:, None, :]
    us = x["q"][idx_w][:, None, :]
    states = forward_family(alpha, beta, k, v, xs, us, dS_final)
    return [states[T - t] for t in range(T)]  # G_s = dS_{T-1-s}, s = T - 1 - t


def test_cotangent_carry_is_the_forward_family_reversed():
    _, x, dout, dS_final = case()
    seq = adjoint_sequential(x, dout, dS_final)
    rev = adjoint_as_forward(x, dout, dS_final)
    for t in range(len(seq)):
        np.testing.assert_allclose(rev[t], seq[t], rtol=1e-12, atol=1e-12)


def chunk_backward(x, X, dout, S_in, G_end, t0, t1):
    """The token-serial backward of tokens [t0, t1) alone, from the state entering the chunk and
    the cotangent of its last state.  Returns per-token dq, dk, dbeta, dalpha, du, dx, z."""
    k, q, v, u, al, be = x["k"], x["q"], x["v"], x["u"], x["alpha"], x["beta"]
    states = forward_family(al[t0:t1], be[t0:t1], k[t0:t1], v[t0:t1], X[t0:t1], u[t0:t1], S_in)
    n = t1 - t0
    R = X.shape[1]
    g = {"dq": np.zeros((n, q.shape[1])), "dk": np.zeros((n, k.shape[1])), "dbeta": np.zeros(n),
         "dalpha": np.zeros(n), "du": np.zeros((n, R, k.shape[1])), "dx": np.zeros((n, R, v.shape[1])),
         "z": np.zeros((n, v.shape[1]))}
    G = G_end
    for j in range(n - 1, -1, -1):
        t = t0 + j
        P, St = states[j], states[j + 1]
        if j < n - 1:  # carry from token t + 1 and add this token's readout
            kk = k[t + 1]
            G = al[t + 1] * (G - be[t + 1] * np.outer(G @ kk, kk)) + np.outer(dout[t], q[t])
        g["dq"][j] = St.T @ dout[t]
        y, z = P @ k[t], G @ k[t]
        g["z"][j] = z
        g["dbeta"][j] = v[t] @ z - al[t] * (y @ z)
        g["dalpha"][j] = np.sum(G * P) - be[t] * (y @ z)
        g["dk"][j] = G.T @ (be[t] * v[t] - al[t] * be[t] * y) - al[t] * be[t] * (P.T @ z)
        for l in range(R):
            g["dx"][j, l] = G @ u[t, l]
            g["du"][j, l] = G.T @ X[t, l]
    return g


@pytest.mark.parametrize("T", [64, 200, 257])
def test_chunks_from_boundary_values_give_the_oracle_cotangents(T):
    inp, x, dout, dS_final = case(T=T)
    X = factors(x["v"], x["conv_w"], x["gamma"], x["eta"])
    S_all = forward_family(x["alpha"], x["beta"], x["k"], x["v"], X, x["u"], np.zeros((x["v"].shape[1], x["k"].shape[1])))
    G_all = adjoint_as_forward(x, dout, dS_final)
    parts = [chunk_backward(x, X, dout, S_all[t0], G_all[min(t0 + C, T) - 1], t0, min(t0 + C, T))
             for t0 in range(0, T, C)]  # every chunk on its own
    got = {kk: np.concatenate([p[kk] for p in parts]) for kk in parts[0]}
    ref = prism_backward.backward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"], inp["gamma"],
                                  inp["eta"], inp["conv_w"], inp["L"], dout[None, None],
                                  dS_final=dS_final[None, None], nthreads=1)
    for name in ("dq", "dk", "dbeta", "dalpha", "du"):
        np.testing.assert_allclose(got[name], ref[name][0, 0], rtol=1e-9, atol=1e-11, err_msg=name)
    # the rest is token-local given dx and z: the chain and convolution backwards
    tail = chain_and_conv_backward(x, got["dx"], got["z"])
    for name in ("dv", "dgamma", "deta", "dconv_w"):
        r = ref[name][0, 0] if name != "dconv_w" else ref[name][0]
        np.testing.assert_allclose(tail[name], r, rtol=1e-9, atol=1e-11, err_msg=name)


def chain_and_conv_backward(x, dx, z):
    """dv = beta z + the residual chain's and the convolution's shares; dgamma, deta, dconv_w."""
    from scipy.special import ndtr
    v, w, gam, eta, beta = x["v"], x["conv_w"], x["gamma"], x["eta"], x["beta"]
    T, dv = v.shape
    R = gam.shape[1]
    h = np.zeros_like(v)
    for j in range(4):
        h[j:] += w[j] * v[: T - j]
    Phi, phi = ndtr(h), np.exp(-h * h / 2) / np.sqrt(2 * np.pi)
    g = Phi + h * phi
    r = [v - h * Phi]
    for l in range(R - 1):
        r.append(r[-1] * (1 - eta[:, l, None] * g))
    out = {"dv": beta[:, None] * z, "dgamma": np.zeros((T, R)), "deta": np.zeros((T, R))}
    drn, dg = np.zeros_like(v), np.zeros_like(v)
    for l in range(R - 1, -1, -1):
        out["dgamma"][:, l] = np.sum(g * r[l] * dx[:, l], axis=1)
        out["deta"][:, l] = -np.sum(g * r[l] * drn, axis=1)
        dg = dg + gam[:, l, None] * r[l] * dx[:, l] - eta[:, l, None] * r[l] * drn
        drn = gam[:, l, None] * g * dx[:, l] + (1 - eta[:, l, None] * g) * drn
    out["dv"] = out["dv"] + drn
    dh = -g * drn + phi * (2 - h * h) * dg
    out["dconv_w"] = np.zeros((4, dv))
    for j in range(4):
        out["dv"][: T - j] += w[j] * dh[j:]
        out["dconv_w"][j] = np.sum(dh[j:] * v[: T - j], axis=0)
    return out
