"""The chunk-map arrangement of the backward pass, in fp64 on the CPU, against the backward oracle.

The backward's two carried quantities -- the state S entering every 64-token chunk and the
cotangent G flowing into every chunk's last state from later tokens -- obey chunk-level affine
recurrences with input-only maps (notes on PRISM, section 2.1, the associative form of the state
passing; section 2.2 for the delta-rule transition alpha (I - beta k k^T)):
    S_{c+1} = S_c A_c + B_c,        G_{c-1} = G_c A_c^T + Bbar_c,
with A_c the chunk's product of transitions (symmetric factors, so the cotangent runs through its
transpose).  With a chunk's WY factors (T = (I + diag(beta) Akk)^{-1}, W = T diag(beta Gamma) K,
U' = T diag(beta) E0 with E0 = V - sum_l Mku_l X_l) and colf_j = Gamma_n / Gamma_j:
    A_c    = Gamma_n I - W^T diag(colf) K
    B_c    = U'^T diag(colf) K + sum_l X_l^T diag(colf) U_l
    Bbar_c = dO^T diag(Gamma) Q - Z0^T diag(beta Gamma) K,    Z0 = T^T (Q K^T o D_incl)^T dO.
Given S_c and G_c, every per-token cotangent of the chunk is a handful of chunk-sized products:
    Vt = U' - W S_c^T                         (the delta-rule values, forward)
    Z  = Z0 + Wbar G_c^T,  Wbar = T^T diag(colf) K      (z_t = G_t k_t, the cotangent of Vt)
    dX_l = diag(colf) U_l G_c^T + P_l^T dO - Mku_l^T diag(beta) Z
    J = (Vw dO^T) o Dbar_incl,  H = (Vw Z^T) o Dbar_strict,   Vw = [Vt; X_1; ...; X_R]
    dKw = diag(colf) Vw G_c + J Q - H diag(beta) K            (rows: dk's write part, du_l)
    dq  = diag(Gamma) dO S_c + J^T Kw,   dk = dKw_0 - diag(beta) (diag(Gamma) Z S_c + H^T Kw)
    dbeta = rowsum(Z o (E - Akk Vt)),  E = E0 - diag(Gamma) K S_c^T
    alpha_t dalpha_t = <G_c, S_{c+1}> + sum_{j >= t in chunk} (q_j.dq_j - beta_j v_j.z_j - sum_l x_jl.dx_jl)
where Akk = K K^T o D_strict, Mku_l = K U_l^T o D_strict, P_l = Q U_l^T o D_incl, Kw = [K; U_1; ...],
D_ij = e^{lambda_i - lambda_j}.  This file restates those steps in numpy and checks that they give
every cotangent of the fp64 backward oracle, including the initial-state and history inputs, a
ragged last chunk and L = 1.  The GPU's chunk-map backward follows the same steps.
"""
import numpy as np
import pytest

from oracle import prism_backward
from ssm_sequence_layer_gb300.inputs import make_cotangents, make_inputs

C = 64


def gelu_parts(h):
    from scipy.special import ndtr
    Phi = ndtr(h)
    phi = np.exp(-h * h / 2) / np.sqrt(2 * np.pi)
    return Phi, phi


def factors_with_history(v, vh, w, gamma, eta):
    """x_{t,l} = gamma g r_l with the anchor reading the three history tokens before t = 0."""
    T, dv = v.shape
    ext = np.concatenate([vh, v], axis=0)  # [3 + T, dv]
    h = np.zeros_like(v)
    for j in range(4):
        h += w[j] * ext[3 - j: 3 - j + T]
    Phi, phi = gelu_parts(h)
    g = Phi + h * phi
    r = v - h * Phi
    R = gamma.shape[1]
    X = np.zeros((T, R, dv))
    for l in range(R):
        X[:, l] = gamma[:, l, None] * g * r
        r = r * (1 - eta[:, l, None] * g)
    return X


def chunk_pieces(q, k, v, u, beta, alpha, X, dO):
    """Per-chunk quantities that depend on the chunk's inputs only (the first kernel): the maps
    A_c, B_c, Bbar_c and the factors the gradient step reuses.  n <= 64 tokens, padded to 64
    with identity tokens (alpha = 1, beta = 0, zero vectors)."""
    n = len(alpha)
    pad = C - n
    P2 = lambda a: np.concatenate([a, np.zeros((pad,) + a.shape[1:])]) if pad else a
    q, k, v, u, X, dO = P2(q), P2(k), P2(v), P2(u), P2(X), P2(dO)
    beta = np.concatenate([beta, np.zeros(pad)])
    alpha = np.concatenate([alpha, np.ones(pad)])
    R = u.shape[1]
    lam = np.cumsum(np.log(alpha))
    Gam = np.exp(lam)
    colf = np.exp(lam[-1] - lam)
    Dm = np.exp(lam[:, None] - lam[None, :])
    i, j = np.indices((C, C))
    Ds = np.where(j < i, Dm, 0.0)
    Di = np.where(j <= i, Dm, 0.0)
    Akk = (k @ k.T) * Ds
    Mku = [(k @ u[:, l].T) * Ds for l in range(R)]
    Pk = (q @ k.T) * Di
    T = np.linalg.inv(np.eye(C) + beta[:, None] * Akk)
    E0 = v - sum((Mku[l] @ X[:, l] for l in range(R)), np.zeros_like(v))
    Up = T @ (beta[:, None] * E0)
    W = T @ ((beta * Gam)[:, None] * k)
    Y = Pk.T @ dO
    Z0 = T.T @ Y
    Wbar = T.T @ (colf[:, None] * k)
    A = Gam[-1] * np.eye(k.shape[1]) - W.T @ (colf[:, None] * k)
    Bm = Up.T @ (colf[:, None] * k) + sum((X[:, l].T @ (colf[:, None] * u[:, l]) for l in range(R)),
                                          np.zeros((v.shape[1], k.shape[1])))
    Bbar = dO.T @ (Gam[:, None] * q) - Z0.T @ ((beta * Gam)[:, None] * k)
    return dict(A=A, B=Bm, Bbar=Bbar, Up=Up, W=W, Wbar=Wbar, Z0=Z0, E0=E0, n=n)


def chunk_grads(q, k, v, u, beta, alpha, X, dO, pc, S0, G, S1):
    """Per-token cotangents of one chunk from its state S0, the cotangent G flowing into its last
    state from later tokens, and the state S1 after its last token (the second kernel)."""
    n = pc["n"]
    pad = C - n
    P2 = lambda a: np.concatenate([a, np.zeros((pad,) + a.shape[1:])]) if pad else a
    q, k, v, u, X, dO = P2(q), P2(k), P2(v), P2(u), P2(X), P2(dO)
    beta = np.concatenate([beta, np.zeros(pad)])
    alpha_p = np.concatenate([alpha, np.ones(pad)])
    R = u.shape[1]
    lam = np.cumsum(np.log(alpha_p))
    Gam = np.exp(lam)
    colf = np.exp(lam[-1] - lam)
    Dm = np.exp(lam[:, None] - lam[None, :])
    i, j = np.indices((C, C))
    Ds = np.where(j < i, Dm, 0.0)
    Di = np.where(j <= i, Dm, 0.0)
    Akk = (k @ k.T) * Ds
    Mku = [(k @ u[:, l].T) * Ds for l in range(R)]
    Pu = [(q @ u[:, l].T) * Di for l in range(R)]
    Vt = pc["Up"] - pc["W"] @ S0.T
    E = pc["E0"] - Gam[:, None] * (k @ S0.T)
    Z = pc["Z0"] + pc["Wbar"] @ G.T
    dX = [colf[:, None] * (u[:, l] @ G.T) + Pu[l].T @ dO - Mku[l].T @ (beta[:, None] * Z) for l in range(R)]
    Vw = [Vt] + [X[:, l] for l in range(R)]
    Kw = [k] + [u[:, l] for l in range(R)]
    # J[m, j] = (w_m . dout_j) D_{j, m} for j >= m;  H[m, j] = (w_m . z_j) D_{j, m} for j > m
    J = [(vw @ dO.T) * Di.T for vw in Vw]
    Hm = [(vw @ Z.T) * Ds.T for vw in Vw]
    dKw = [colf[:, None] * (Vw[b] @ G) + J[b] @ q - Hm[b] @ (beta[:, None] * k) for b in range(R + 1)]
    dq = Gam[:, None] * (dO @ S0) + sum(J[b].T @ Kw[b] for b in range(R + 1))
    extra = Gam[:, None] * (Z @ S0) + sum(Hm[b].T @ Kw[b] for b in range(R + 1))
    dk = dKw[0] - beta[:, None] * extra
    dbeta = np.sum(Z * (E - Akk @ Vt), axis=1)
    s = np.sum(q * dq, axis=1) - beta * np.sum(v * Z, axis=1)
    for l in range(R):
        s = s - np.sum(X[:, l] * dX[l], axis=1)
    suffix = np.cumsum(s[::-1])[::-1]
    dalpha = (np.sum(G * S1) + suffix) / alpha_p
    out = dict(dq=dq[:n], dk=dk[:n], dbeta=dbeta[:n], dalpha=dalpha[:n], z=Z[:n],
               du=np.stack([dKw[1 + l][:n] for l in range(R)], axis=1) if R else np.zeros((n, 0, k.shape[1])),
               dx=np.stack([d[:n] for d in dX], axis=1) if R else np.zeros((n, 0, v.shape[1])))
    return out


def chunked_backward(x, dout, dS_final, S_init, vh):
    T, dv = x["v"].shape
    dk = x["k"].shape[1]
    R = x["u"].shape[1]
    X = factors_with_history(x["v"], vh, x["conv_w"], x["gamma"], x["eta"]) if R else np.zeros((T, 0, dv))
    NC = (T + C - 1) // C
    sl = [slice(c * C, min(T, c * C + C)) for c in range(NC)]
    pcs = [chunk_pieces(x["q"][s], x["k"][s], x["v"][s], x["u"][s], x["beta"][s], x["alpha"][s], X[s], dout[s])
           for s in sl]
    S = [S_init]
    for c in range(NC):
        S.append(S[-1] @ pcs[c]["A"] + pcs[c]["B"])
    G = [None] * NC
    g = dS_final
    for c in range(NC - 1, -1, -1):
        G[c] = g
        g = g @ pcs[c]["A"].T + pcs[c]["Bbar"]
    dS_init = g
    parts = [chunk_grads(x["q"][s], x["k"][s], x["v"][s], x["u"][s], x["beta"][s], x["alpha"][s], X[s], dout[s],
                         pcs[c], S[c], G[c], S[c + 1]) for c, s in enumerate(sl)]
    got = {kk: np.concatenate([p[kk] for p in parts]) for kk in parts[0]}
    got["dS_init"] = dS_init
    got["S_final"] = S[-1]
    return got


def case(T, L, dk=16, dv=12, seed=3, state=True):
    inp = make_inputs(1, 1, T, dk, dv, L, dtype="f32", seed=seed)
    x = {n: inp[n].double().numpy()[0, 0] for n in ("q", "k", "v", "beta", "alpha")}
    R = L - 1
    if R:
        for n in ("u", "gamma", "eta"):
            x[n] = inp[n].double().numpy()[0, 0]
    else:
        x["u"] = np.zeros((T, 0, dk))
        x["gamma"] = np.zeros((T, 0))
        x["eta"] = np.zeros((T, 0))
    x["conv_w"] = inp["conv_w"].double().numpy()[0]
    dout, dS_final = make_cotangents(1, 1, T, dk, dv, seed=seed, with_state=True)
    g = np.random.default_rng(seed)
    S_init = 0.3 * g.standard_normal((dv, dk)) if state else np.zeros((dv, dk))
    vh = g.standard_normal((3, dv)) if state else np.zeros((3, dv))
    return inp, x, dout.double().numpy()[0, 0], (dS_final.double().numpy()[0, 0] if state else np.zeros((dv, dk))), \
        S_init, vh


@pytest.mark.parametrize("T,L,state", [(64, 3, False), (200, 3, True), (257, 4, True), (130, 1, True), (45, 2, True)])
def test_chunk_maps_give_the_oracle_cotangents(T, L, state):
    inp, x, dout, dS_final, S_init, vh = case(T, L, state=state)
    got = chunked_backward(x, dout, dS_final, S_init, vh)
    ref = prism_backward.backward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"], inp["gamma"],
                                  inp["eta"], inp["conv_w"], inp["L"], dout[None, None],
                                  S_init=S_init[None, None], v_hist=vh[None, None], dS_final=dS_final[None, None],
                                  want_dv_hist=True, want_dS_init=True, nthreads=1)
    names = ["dq", "dk", "dbeta", "dalpha"] + (["du"] if L > 1 else [])
    for name in names:
        np.testing.assert_allclose(got[name], ref[name][0, 0], rtol=1e-9, atol=1e-10, err_msg=name)
    np.testing.assert_allclose(got["dS_init"], ref["dS_init"][0, 0], rtol=1e-9, atol=1e-10, err_msg="dS_init")
    if L > 1:
        tail = chain_and_conv_backward_hist(x, vh, got["dx"], got["z"])
        for name in ("dv", "dgamma", "deta", "dconv_w", "dv_hist"):
            r = ref[name][0, 0] if name != "dconv_w" else ref[name][0]
            np.testing.assert_allclose(tail[name], r, rtol=1e-9, atol=1e-10, err_msg=name)
    else:
        np.testing.assert_allclose(x["beta"][:, None] * got["z"], ref["dv"][0, 0], rtol=1e-9, atol=1e-10)


def chain_and_conv_backward_hist(x, vh, dx, z):
    """chain_and_conv_backward with the anchor reading history tokens (their cotangent returned)."""
    from scipy.special import ndtr
    v, w, gam, eta, beta = x["v"], x["conv_w"], x["gamma"], x["eta"], x["beta"]
    T, dv = v.shape
    R = gam.shape[1]
    ext = np.concatenate([vh, v], axis=0)
    h = np.zeros_like(v)
    for j in range(4):
        h += w[j] * ext[3 - j: 3 - j + T]
    Phi, phi = ndtr(h), np.exp(-h * h / 2) / np.sqrt(2 * np.pi)
    g = Phi + h * phi
    r = [v - h * Phi]
    for l in range(R - 1):
        r.append(r[-1] * (1 - eta[:, l, None] * g))
    out = {"dgamma": np.zeros((T, R)), "deta": np.zeros((T, R))}
    drn, dg = np.zeros_like(v), np.zeros_like(v)
    for l in range(R - 1, -1, -1):
        out["dgamma"][:, l] = np.sum(g * r[l] * dx[:, l], axis=1)
        out["deta"][:, l] = -np.sum(g * r[l] * drn, axis=1)
        dg = dg + gam[:, l, None] * r[l] * dx[:, l] - eta[:, l, None] * r[l] * drn
        drn = gam[:, l, None] * g * dx[:, l] + (1 - eta[:, l, None] * g) * drn
    dh = -g * drn + phi * (2 - h * h) * dg
    dext = np.zeros_like(ext)
    dext[3:] = beta[:, None] * z + drn
    out["dconv_w"] = np.zeros((4, dv))
    for j in range(4):
        dext[3 - j: 3 - j + T] += w[j] * dh
        out["dconv_w"][j] = np.sum(dh * ext[3 - j: 3 - j + T], axis=0)
    out["dv"] = dext[3:]
    out["dv_hist"] = dext[:3]
    return out


def test_chunk_maps_reproduce_the_forward_final_state():
    """S_{c+1} = S_c A_c + B_c over all chunks gives the oracle's final state."""
    from oracle import prism_oracle
    inp, x, dout, dS_final, S_init, vh = case(200, 3, state=True)
    got = chunked_backward(x, dout, dS_final, S_init, vh)
    ref = prism_oracle.forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"], inp["gamma"],
                               inp["eta"], inp["conv_w"], inp["L"], S_init=S_init[None, None], v_hist=vh[None, None],
                               want_state=True, nthreads=1)
    np.testing.assert_allclose(got["S_final"], np.asarray(ref["S_final"])[0, 0], rtol=1e-10, atol=1e-12)


def exact_dalpha(q, k, v, u, beta, alpha, X, dO, pc, S0, G, Vt, Z):
    """alpha_t dalpha_t = <G_t, alpha_t S_{t-1}> - beta_t z_t . yhat_t from the chunk's quantities with
    no cancellation: every term carries a decay that spans token t.  With writes w = (tau_w,
    omega_w, kappa_w) (Vt_tau k_tau^T and x_tau,l u_tau,l^T), Gamma_t = e^{lambda_t}, n the chunk's
    last token:
      T1 = Gamma_n <G, S0>                       T2_t = sum_{tau_w < t} colf_tau omega_w . G kappa_w
      T3_t = sum_{j >= t} Gamma_j dout_j . S0 q_j
      T4_t = sum_{j >= t > tau_w} D_{j,tau_w} (dout_j . omega_w)(q_j . kappa_w)
      T5_t = -sum_{j > t} Gamma_j beta_j z_j . S0 k_j
      T6_t = -sum_{j > t > tau_w} D_{j,tau_w} beta_j (z_j . omega_w)(k_j . kappa_w)
      yhat_t = alpha_t S_{t-1} k_t = v_t - Vt_t / beta_t ... formed as Gamma_t S0 k_t + sum_{tau_w < t}
               D_{t,tau_w} (kappa_w . k_t) omega_w (no division)."""
    n = pc["n"]
    pad = C - n
    P2 = lambda a: np.concatenate([a, np.zeros((pad,) + a.shape[1:])]) if pad else a
    q, k, v, u, X, dO = P2(q), P2(k), P2(v), P2(u), P2(X), P2(dO)
    beta = np.concatenate([beta, np.zeros(pad)])
    alpha_p = np.concatenate([alpha, np.ones(pad)])
    R = u.shape[1]
    lam = np.cumsum(np.log(alpha_p))
    Gam = np.exp(lam)
    colf = np.exp(lam[-1] - lam)
    Dm = np.exp(lam[:, None] - lam[None, :])
    Vw = [Vt] + [X[:, l] for l in range(R)]
    Kw = [k] + [u[:, l] for l in range(R)]
    a = sum(np.sum(Vw[b] * (Kw[b] @ G.T), axis=1) for b in range(R + 1))   # omega_w . G kappa_w per token
    bq = np.sum(dO * (q @ S0.T), axis=1)                                   # dout_j . S0 q_j
    dz = np.sum(Z * (k @ S0.T), axis=1)                                    # z_j . S0 k_j
    T1 = Gam[-1] * np.sum(G * S0)
    idx = np.arange(C)
    T2 = np.array([np.sum(colf[:t] * a[:t]) for t in range(C)])
    T3 = np.array([np.sum(Gam[t:] * bq[t:]) for t in range(C)])
    T5 = -np.array([np.sum((Gam * beta * dz)[t + 1:]) for t in range(C)])
    T4 = np.zeros(C)
    T6 = np.zeros(C)
    for b in range(R + 1):
        Cm = (dO @ Vw[b].T) * (q @ Kw[b].T) * np.where(idx[:, None] > idx[None, :], Dm, 0.0)   # [j][tau]
        Em = (Z @ Vw[b].T) * (k @ Kw[b].T) * beta[:, None] * np.where(idx[:, None] > idx[None, :], Dm, 0.0)
        for t in range(C):
            T4[t] += np.sum(Cm[t:, :t])
            T6[t] -= np.sum(Em[t + 1:, :t])
    yhat = Gam[:, None] * (k @ S0.T) + sum(((k @ Kw[b].T) * np.where(idx[:, None] > idx[None, :], Dm, 0.0)) @ Vw[b]
                                            for b in range(R + 1))
    num = T1 + T2 + T3 + T4 + T5 + T6 - beta * np.sum(Z * yhat, axis=1)
    return (num / alpha_p)[:n]


@pytest.mark.parametrize("alpha_div", [16.0, 0.25])
def test_exact_dalpha_from_the_chunk_terms(alpha_div):
    """The cancellation-free dalpha agrees with the oracle, including gates far below one where the
    suffix-sum identity loses its precision."""
    T, L = 200, 4
    inp = make_inputs(1, 1, T, 16, 12, L, dtype="f32", seed=5, alpha_div=alpha_div)
    x = {nm: inp[nm].double().numpy()[0, 0] for nm in ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")}
    x["conv_w"] = inp["conv_w"].double().numpy()[0]
    dout, dS_final = make_cotangents(1, 1, T, 16, 12, seed=5, with_state=True)
    dout, dS_final = dout.double().numpy()[0, 0], dS_final.double().numpy()[0, 0]
    g = np.random.default_rng(5)
    S_init, vh = 0.3 * g.standard_normal((12, 16)), g.standard_normal((3, 12))
    X = factors_with_history(x["v"], vh, x["conv_w"], x["gamma"], x["eta"])
    NC = (T + C - 1) // C
    sl = [slice(c * C, min(T, c * C + C)) for c in range(NC)]
    pcs = [chunk_pieces(x["q"][s], x["k"][s], x["v"][s], x["u"][s], x["beta"][s], x["alpha"][s], X[s], dout[s])
           for s in sl]
    S = [S_init]
    for c in range(NC):
        S.append(S[-1] @ pcs[c]["A"] + pcs[c]["B"])
    Gs = [None] * NC
    gg = dS_final
    for c in range(NC - 1, -1, -1):
        Gs[c] = gg
        gg = gg @ pcs[c]["A"].T + pcs[c]["Bbar"]
    got = []
    for c, s in enumerate(sl):
        pc = pcs[c]
        n = pc["n"]
        pad = C - n
        P2 = lambda a: np.concatenate([a, np.zeros((pad,) + a.shape[1:])]) if pad else a
        Vt = pc["Up"] - pc["W"] @ S[c].T
        Z = pc["Z0"] + pc["Wbar"] @ Gs[c].T
        got.append(exact_dalpha(x["q"][s], x["k"][s], x["v"][s], x["u"][s], x["beta"][s], x["alpha"][s], X[s],
                                dout[s], pc, S[c], Gs[c], Vt, Z))
    got = np.concatenate(got)
    ref = prism_backward.backward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"], inp["gamma"],
                                  inp["eta"], inp["conv_w"], inp["L"], dout[None, None], S_init=S_init[None, None],
                                  v_hist=vh[None, None], dS_final=dS_final[None, None], nthreads=1)
    np.testing.assert_allclose(got, ref["dalpha"][0, 0], rtol=1e-8, atol=1e-10)
