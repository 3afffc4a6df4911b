"""Pins for the fp64 backward oracle: its cotangents against central finite differences of
the forward oracle (itself pinned in test_oracle_pins.py).

The backward is reverse-mode differentiation of the sequential definition (notes on PRISM,
sections 2.2-2.3; Tencent article, part 03).  A derivative has a plain definition: the limit
of the forward's difference quotients.  So each test perturbs one input of the forward
oracle along a random direction D and compares

    (f(x + eps D) - f(x - eps D)) / (2 eps)   with   <dLoss/dx, D>,

where f = <dout, out> + <dS_final, S_final>.  In fp64 with eps = 1e-5 the central difference
is exact to about 1e-9 relative (the truncation term is eps^2 times a third derivative of
smooth functions: exp, erf, products).  A dropped term, a wrong sign, a wrong index or a
transposed operand anywhere in the backward changes the inner product by far more.
The tiny case also compares every element of every cotangent with its own difference quotient.
"""
import numpy as np
import pytest

from oracle import prism_backward, prism_oracle
from ssm_sequence_layer_gb300.inputs import make_cotangents, make_gain, make_inputs

INPUT_NAMES = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta", "conv_w")


def f64_case(B=1, H=2, T=24, dk=6, dv=5, L=3, seed=3, state=True, hist=True, nonlinear=False):
    """Inputs of one case; with `nonlinear` the forward is the non-linear residual variant:
    gains p (make_gain) take the place of eta."""
    inp = make_inputs(B, H, T, dk, dv, L, dtype="f32", seed=seed)
    x = {n: inp[n].double().numpy() for n in INPUT_NAMES}
    x["p_gain"] = make_gain(B, H, T, L, dv, dtype="f32", seed=seed).double().numpy() if nonlinear else None
    if nonlinear:
        x["eta"] = None
    rng = np.random.default_rng(seed + 11)
    x["S_init"] = rng.standard_normal((B, H, dv, dk)) * 0.3 if state else None
    x["v_hist"] = rng.standard_normal((B, H, 3, dv)) if hist else None
    dout, dS_final = make_cotangents(B, H, T, dk, dv, seed=seed, with_state=state)
    cot = {"dout": dout.double().numpy(), "dS_final": dS_final.double().numpy() if state else None}
    return x, cot, L


def loss(x, cot, L):
    r = prism_oracle.forward(x["q"], x["k"], x["v"], x["beta"], x["alpha"], x["u"], x["gamma"], x["eta"],
                             x["conv_w"], L, S_init=x["S_init"], v_hist=x["v_hist"], p_gain=x.get("p_gain"),
                             want_state=True, nthreads=1)
    f = float(np.sum(cot["dout"] * r["out"]))
    if cot["dS_final"] is not None:
        f += float(np.sum(cot["dS_final"] * r["S_final"]))
    return f


def grads(x, cot, L, mod=prism_backward):
    return mod.backward(x["q"], x["k"], x["v"], x["beta"], x["alpha"], x["u"], x["gamma"], x["eta"], x["conv_w"],
                        L, cot["dout"], S_init=x["S_init"], v_hist=x["v_hist"], dS_final=cot["dS_final"],
                        p_gain=x.get("p_gain"), want_dv_hist=True, want_dS_init=True, nthreads=1)


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "alpha": "dalpha", "u": "du", "gamma": "dgamma",
           "eta": "deta", "conv_w": "dconv_w", "S_init": "dS_init", "v_hist": "dv_hist", "p_gain": "dp_gain"}


def directional_check(x, cot, L, name, g, eps=1e-5, seed=0):
    """|<g, D> - central difference| relative to the size of the terms."""
    rng = np.random.default_rng(seed)
    D = rng.standard_normal(x[name].shape)
    xp = dict(x)
    xm = dict(x)
    xp[name] = x[name] + eps * D
    xm[name] = x[name] - eps * D
    fd = (loss(xp, cot, L) - loss(xm, cot, L)) / (2 * eps)
    an = float(np.sum(g[GRAD_OF[name]] * D))
    scale = float(np.sqrt(np.sum(g[GRAD_OF[name]] ** 2) * np.sum(D ** 2))) + 1e-30
    return abs(an - fd) / scale, an, fd


ALL = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta", "conv_w", "S_init", "v_hist")


def inputs_of(x):
    """The differentiable inputs present in a case (eta or p_gain, S_init and v_hist if given)."""
    names = [n for n in ALL if x.get(n) is not None]
    return names + (["p_gain"] if x.get("p_gain") is not None else [])


@pytest.mark.parametrize("L", [1, 2, 4])
def test_directional_derivatives_match_central_differences(L):
    x, cot, L = f64_case(L=L, T=21, B=2, H=2)
    g = grads(x, cot, L)
    for name in ALL:
        if L == 1 and name in ("u", "gamma", "eta"):
            continue
        for seed in (0, 1):
            err, an, fd = directional_check(x, cot, L, name, g, seed=seed)
            assert err < 1e-8, f"d/d{name} (L={L}): analytic {an!r} vs central difference {fd!r}"


def test_every_element_on_a_tiny_case():
    """Each cotangent entry against its own difference quotient (B=1, H=1, T=6, dk=3, dv=2, L=3)."""
    x, cot, L = f64_case(B=1, H=1, T=6, dk=3, dv=2, L=3, seed=5)
    g = grads(x, cot, L)
    eps = 1e-6
    for name in ALL:
        gx = g[GRAD_OF[name]]
        flat = x[name].reshape(-1)
        for idx in range(flat.size):
            xp = dict(x)
            xm = dict(x)
            a = flat.copy()
            a[idx] += eps
            xp[name] = a.reshape(x[name].shape)
            b = flat.copy()
            b[idx] -= eps
            xm[name] = b.reshape(x[name].shape)
            fd = (loss(xp, cot, L) - loss(xm, cot, L)) / (2 * eps)
            assert abs(gx.reshape(-1)[idx] - fd) <= 1e-7 * (1 + abs(fd)), (name, idx, gx.reshape(-1)[idx], fd)


def test_unread_gain_slot_is_never_read():
    """eta[..., R-1] shapes a residual nothing uses: NaN there changes no cotangent."""
    x, cot, L = f64_case(L=3)
    g = grads(x, cot, L)
    x2 = dict(x)
    x2["eta"] = x["eta"].copy()
    x2["eta"][..., L - 2] = np.nan
    g2 = grads(x2, cot, L)
    for key in g:
        assert np.array_equal(g[key], g2[key]), key


def test_unread_gain_slot_has_zero_cotangent():
    x, cot, L = f64_case(L=3)
    g = grads(x, cot, L)
    assert np.all(g["deta"][..., L - 2] == 0.0)
    assert np.any(g["deta"][..., 0] != 0.0)


def test_dq_is_the_transposed_state_times_dout():
    """dq_t = S_t^T dout_t, with S_t the forward oracle's final state of the prefix 0..t."""
    x, cot, L = f64_case(B=1, H=1, T=9, L=3, state=False, hist=False)
    g = grads(x, cot, L)
    for t in (0, 4, 8):
        pre = {n: (x[n][:, :, : t + 1] if n not in ("conv_w",) else x[n]) for n in INPUT_NAMES}
        r = prism_oracle.forward(pre["q"], pre["k"], pre["v"], pre["beta"], pre["alpha"], pre["u"], pre["gamma"],
                                 pre["eta"], pre["conv_w"], L, want_state=True, nthreads=1)
        St = r["S_final"][0, 0]
        np.testing.assert_allclose(g["dq"][0, 0, t], St.T @ cot["dout"][0, 0, t], rtol=1e-12, atol=1e-12)


def test_zero_cotangents_give_zero_gradients():
    x, cot, L = f64_case(L=3)
    cot = {"dout": np.zeros_like(cot["dout"]), "dS_final": np.zeros_like(cot["dS_final"])}
    g = grads(x, cot, L)
    for key, val in g.items():
        assert np.all(val == 0.0), key


def test_gradients_are_linear_in_the_cotangents():
    x, cot, L = f64_case(L=2)
    g1 = grads(x, cot, L)
    cot2 = {"dout": 2.5 * cot["dout"], "dS_final": 2.5 * cot["dS_final"]}
    g2 = grads(x, cot2, L)
    for key in g1:
        np.testing.assert_allclose(g2[key], 2.5 * g1[key], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("L", [2, 4])
def test_nonlinear_variant_directional_derivatives(L):
    """The non-linear residual variant (gains p in place of eta): every input, p included."""
    x, cot, L = f64_case(L=L, T=21, B=2, H=2, nonlinear=True)
    g = grads(x, cot, L)
    assert "deta" not in g and g["dp_gain"].shape == x["p_gain"].shape
    for name in inputs_of(x):
        for seed in (0, 1):
            err, an, fd = directional_check(x, cot, L, name, g, seed=seed)
            assert err < 1e-8, f"d/d{name} (non-linear, L={L}): analytic {an!r} vs central difference {fd!r}"


def test_nonlinear_variant_every_element_on_a_tiny_case():
    x, cot, L = f64_case(B=1, H=1, T=6, dk=3, dv=2, L=3, seed=7, nonlinear=True)
    g = grads(x, cot, L)
    eps = 1e-6
    for name in inputs_of(x):
        gx = g[GRAD_OF[name]].reshape(-1)
        flat = x[name].reshape(-1)
        for idx in range(flat.size):
            a, b = flat.copy(), flat.copy()
            a[idx] += eps
            b[idx] -= eps
            fd = (loss(dict(x, **{name: a.reshape(x[name].shape)}), cot, L)
                  - loss(dict(x, **{name: b.reshape(x[name].shape)}), cot, L)) / (2 * eps)
            assert abs(gx[idx] - fd) <= 1e-7 * (1 + abs(fd)), (name, idx, gx[idx], fd)
