"""Pins for the input-projection oracle (oracle/prism_projection.py): each checks it against a
library routine or a property its definition fixes, chosen so that a slip in the convolution
(tap order, causality, batch leakage), the weight layout (head / level / channel order) or an
activation fails one of them."""
import numpy as np

from oracle import prism_projection as PP


def rand_case(B=2, T=11, D=8, H=2, R=2, dk=4, dv=3, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((B, T, D))
    w = rng.standard_normal((4, D)) * 0.5
    N = H * R * (dk + dv + 1)
    W = rng.standard_normal((N, D)) / np.sqrt(D)
    return X, w, W


def test_anchor_is_numpy_causal_convolution():
    X, w, _ = rand_case()
    a = PP.anchor(X, w)
    for b in range(X.shape[0]):
        for d in range(X.shape[2]):
            ref = np.convolve(X[b, :, d], w[:, d])[: X.shape[1]]
            np.testing.assert_allclose(a[b, :, d], ref, rtol=1e-13, atol=1e-14)


def test_basis_is_unit_and_scale_invariant():
    X, w, W = rand_case()
    H, R, dk, dv = 2, 2, 4, 3
    u, p, g = PP.project(X, w, W, H, R, dk, dv)
    np.testing.assert_allclose(np.linalg.norm(u, axis=-1), 1.0, rtol=1e-13)
    W2 = W.copy()
    W2[: H * R * dk] *= 3.7   # the basis rows only
    u2, p2, g2 = PP.project(X, w, W2, H, R, dk, dv)
    np.testing.assert_allclose(u2, u, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(p2, p)
    W2[: H * R * dk] *= -1.0
    u3, _, _ = PP.project(X, w, W2, H, R, dk, dv)
    np.testing.assert_allclose(u3, -u, rtol=1e-12, atol=1e-14)


def test_gain_is_linear_and_gate_is_a_logistic():
    X, w, W = rand_case(seed=1)
    H, R, dk, dv = 2, 2, 4, 3
    X2 = np.random.default_rng(7).standard_normal(X.shape)
    _, p1, g1 = PP.project(X, w, W, H, R, dk, dv)
    _, p2, _ = PP.project(X2, w, W, H, R, dk, dv)
    _, p12, _ = PP.project(X + X2, w, W, H, R, dk, dv)
    np.testing.assert_allclose(p12, p1 + p2, rtol=1e-12, atol=1e-12)
    Wn = W.copy()
    Wn[-H * R:] *= -1.0       # gate rows negated: sigmoid(-z) = 1 - sigmoid(z)
    _, _, gn = PP.project(X, w, Wn, H, R, dk, dv)
    np.testing.assert_allclose(gn, 1.0 - g1, rtol=1e-12, atol=1e-14)
    Wz = W.copy()
    Wz[-H * R:] = 0.0
    _, _, gz = PP.project(X, w, Wz, H, R, dk, dv)
    assert np.all(gz == 0.5)


def test_weight_layout_by_one_hot_rows():
    """Row (h, l, c) of the gain block picks feature f(h, l, c): p[b, h, t, l, c] must equal the
    anchor's feature f at token t, which fixes the head / level / channel order of every block."""
    B, T, H, R, dk, dv = 1, 5, 2, 3, 2, 2
    D = H * R * dv
    X, w, _ = rand_case(B=B, T=T, D=D, seed=2)
    a = PP.anchor(X, w)
    N = H * R * (dk + dv + 1)
    W = np.zeros((N, D))
    NU = H * R * dk
    for h in range(H):
        for l in range(R):
            for c in range(dv):
                W[NU + (h * R + l) * dv + c, (h * R + l) * dv + c] = 1.0
            W[NU + H * R * dv + h * R + l, (h * R + l) * dv] = 1.0   # gate of (h, l): feature of its first gain row
            W[(h * R + l) * dk, (h * R + l) * dv + 1] = -1.0           # basis of (h, l): minus one feature
    u, p, g = PP.project(X, w, W, H, R, dk, dv)
    for h in range(H):
        for l in range(R):
            f = (h * R + l) * dv
            np.testing.assert_array_equal(p[0, h, :, l, :], a[0, :, f:f + dv])
            np.testing.assert_allclose(g[0, h, :, l], 1 / (1 + np.exp(-a[0, :, f])), rtol=1e-14)
            np.testing.assert_array_equal(u[0, h, :, l, 0], -np.sign(a[0, :, f + 1]))
            assert np.all(u[0, h, :, l, 1:] == 0)


def test_batches_do_not_leak_through_the_convolution():
    X, w, W = rand_case(B=3, seed=3)
    u, p, g = PP.project(X, w, W, 2, 2, 4, 3)
    u1, p1, g1 = PP.project(X[1:2], w, W, 2, 2, 4, 3)
    np.testing.assert_array_equal(p1[0], p[1])
    np.testing.assert_array_equal(g1[0], g[1])
