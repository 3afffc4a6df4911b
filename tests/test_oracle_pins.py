"""Pins for the fp64 oracle: each test checks it against something other than itself.

The pages print no worked numbers for the recurrence, so the oracle is pinned by
closed forms, library routines, brute force and invariants that the method's
definition fixes (notes on PRISM, sections 2.2-2.3; Tencent article, part 03):

  * L = 1 equals an independent delta-form GDN loop (the first step "degenerates
    to the standard GDN write", article part 03 item four);
  * the injection factors equal the closed-form residual chain (article part 03
    item three: the chain is an element-wise linear recursion);
  * for T <= 16 the output equals the explicit product of dense transition
    matrices A_s = alpha_s (I - beta_s k_s k_s^T) and injections B_t (notes,
    section 2.1: S_t = S_{t-1} A_t + B_t with input-only A, B);
  * beta = gamma = 0 gives S = 0; alpha = 1 with orthonormal keys gives exact
    recall; alpha = 1, beta = 0 is causal linear attention with rank-(L-1) writes;
    conv_w = 0 gives h = 0, g = 1/2, e = v;
  * a token's injection has rank min(L, dv, dk) (notes, section 2.5);
  * the anchor is a causal depthwise window of four taps, zero before t = 0;
  * gain and residual match GELU built from scipy's normal CDF, and the gain is
    the derivative of that GELU.
Each of these is chosen so a plausible slip (dropped term, wrong sign, wrong
index or a transposed operand) in the oracle fails at least one of them.
"""
import numpy as np
import pytest
import scipy.special as sps

from ssm_sequence_layer_gb300.inputs import make_inputs


def f64_inputs(B=1, H=2, T=40, dk=8, dv=6, L=3, seed=1, alpha_div=16.0):
    inp = make_inputs(B, H, T, dk, dv, L, dtype="f32", seed=seed, alpha_div=alpha_div)
    out = {kk: (vv.double().numpy() if hasattr(vv, "numpy") else vv) for kk, vv in inp.items()}
    return out


def run(oracle_mod, inp, **kw):
    return oracle_mod.forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"],
                              inp["gamma"], inp["eta"], inp["conv_w"], inp["L"], **kw)


def gelu_lib(x):
    return x * sps.ndtr(x)


def anchor_ref(v, w):
    """h_t = sum_j w_j v_{t-j}, zero before the sequence start; v [B,H,T,dv], w [H,4,dv]."""
    B, H, T, dv = v.shape
    h = np.zeros_like(v)
    for j in range(4):
        h[:, :, j:, :] += w[None, :, j, None, :] * v[:, :, : T - j, :]
    return h


def relerr(a, b):
    return np.max(np.abs(a - b)) / max(np.sqrt(np.mean(b ** 2)), 1e-300)


# ---------------------------------------------------------------------------------------------
def test_gdn_degenerate_equals_delta_rule(oracle_mod):
    inp = f64_inputs(B=2, H=2, T=50, dk=8, dv=5, L=1, seed=3)
    res = run(oracle_mod, inp, want_state=True)
    q, k, v, be, al = inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"]
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    for b in range(B):
        for h in range(H):
            S = np.zeros((dv, dk))
            for t in range(T):
                kt, vt = k[b, h, t], v[b, h, t]
                pred = al[b, h, t] * S @ kt
                S = al[b, h, t] * S + be[b, h, t] * np.outer(vt - pred, kt)
                np.testing.assert_allclose(res["out"][b, h, t], S @ q[b, h, t], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(res["S_final"][b, h], S, rtol=1e-12, atol=1e-13)


def test_gain_and_residual_match_library_gelu(oracle_mod):
    inp = f64_inputs(B=1, H=2, T=30, dk=4, dv=7, L=2, seed=4)
    res = run(oracle_mod, inp, want_hge=True)
    h = anchor_ref(inp["v"], inp["conv_w"])
    np.testing.assert_allclose(res["h"], h, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(res["e"], inp["v"] - gelu_lib(h), rtol=1e-12, atol=1e-13)
    # gain = d/dh GELU(h): 4th-order central difference of the library GELU
    eps = 1e-3
    d = (-gelu_lib(h + 2 * eps) + 8 * gelu_lib(h + eps) - 8 * gelu_lib(h - eps) + gelu_lib(h - 2 * eps)) / (12 * eps)
    np.testing.assert_allclose(res["g"], d, rtol=1e-9, atol=1e-10)


def test_gelu_textbook_points(oracle_mod):
    """GELU(0)=0, GELU'(0)=1/2, and GELU(x) -> x, GELU'(x) -> 1 far right; -> 0 far left."""
    H, dv = 1, 4
    T = 1
    v = np.array([0.0, 1.0, -1.0, 9.0]).reshape(1, 1, 1, dv)
    w = np.zeros((H, 4, dv))
    w[0, 0, :] = 1.0  # h_0 = v_0
    z = np.zeros((1, 1, T))
    q = np.zeros((1, 1, T, 2)); q[..., 0] = 1
    res = oracle_mod.forward(q, q, v, z, np.ones_like(z), None, None, None, w, 1, want_hge=True)
    g, e = res["g"].ravel(), res["e"].ravel()
    assert g[0] == 0.5 and e[0] == 0.0
    np.testing.assert_allclose(1.0 - e[1], sps.ndtr(1.0), rtol=1e-15)      # GELU(1) = Phi(1)
    np.testing.assert_allclose(-1.0 - e[2], -sps.ndtr(-1.0), rtol=1e-15)   # GELU(-1) = -Phi(-1)
    np.testing.assert_allclose(g[1], sps.ndtr(1.0) + np.exp(-0.5) / np.sqrt(2 * np.pi), rtol=1e-15)
    assert abs(e[3]) < 1e-15 and abs(g[3] - 1.0) < 1e-15


def test_anchor_impulse_response(oracle_mod):
    """A unit impulse at t0 reproduces the taps w_0..w_3 at t0..t0+3, per head, nothing across batch."""
    B, H, T, dv = 2, 2, 12, 3
    v = np.zeros((B, H, T, dv))
    v[1, 0, 5, :] = 1.0
    w = np.arange(1, 1 + H * 4 * dv, dtype=float).reshape(H, 4, dv) / 10
    z = np.zeros((B, H, T))
    q = np.zeros((B, H, T, 2)); q[..., 0] = 1
    res = oracle_mod.forward(q, q, v, z, np.ones_like(z), None, None, None, w, 1, want_hge=True)
    h = res["h"]
    expect = np.zeros_like(h)
    for j in range(4):
        expect[1, 0, 5 + j, :] = w[0, j, :]
    assert np.array_equal(h, expect)


def test_residual_chain_closed_form(oracle_mod):
    inp = f64_inputs(B=1, H=2, T=20, dk=4, dv=5, L=6, seed=5)
    res = run(oracle_mod, inp, want_x=True, want_hge=True)
    g, e = res["g"], res["e"]
    gam, eta = inp["gamma"], inp["eta"]
    R = inp["L"] - 1
    factors = 1.0 - eta[..., :, None] * g[..., None, :]          # [B,H,T,R,dv]
    prods = np.cumprod(np.concatenate([np.ones_like(factors[..., :1, :]), factors[..., : R - 1, :]], axis=-2), axis=-2)
    x = gam[..., None] * g[..., None, :] * e[..., None, :] * prods
    np.testing.assert_allclose(res["X"], x, rtol=1e-12, atol=1e-14)


def test_last_eta_slot_is_never_read(oracle_mod):
    inp = f64_inputs(B=1, H=2, T=16, dk=4, dv=4, L=4, seed=6)
    ref = run(oracle_mod, inp)["out"]
    inp["eta"] = inp["eta"].copy()
    inp["eta"][..., -1] = np.nan
    out = run(oracle_mod, inp)["out"]
    assert np.array_equal(out, ref)


def _brute_force(inp):
    """S_t = sum_{tau<=t} B_tau prod_{tau<s<=t} A_s with dense A_s (dk x dk), o_t = S_t q_t."""
    q, k, v, be, al = inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"]
    u, gam, eta, w = inp["u"], inp["gamma"], inp["eta"], inp["conv_w"]
    L = inp["L"]
    R = L - 1
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    h = anchor_ref(v, w)
    g = sps.ndtr(h) + h * np.exp(-h * h / 2) / np.sqrt(2 * np.pi)
    e = v - gelu_lib(h)
    out = np.zeros((B, H, T, dv))
    for b in range(B):
        for hh in range(H):
            A = [al[b, hh, s] * (np.eye(dk) - be[b, hh, s] * np.outer(k[b, hh, s], k[b, hh, s])) for s in range(T)]
            Bm = []
            for s in range(T):
                Bs = be[b, hh, s] * np.outer(v[b, hh, s], k[b, hh, s])
                r = e[b, hh, s].copy()
                for l in range(R):
                    Bs = Bs + gam[b, hh, s, l] * np.outer(g[b, hh, s] * r, u[b, hh, s, l])
                    r = r * (1 - eta[b, hh, s, l] * g[b, hh, s])
                Bm.append(Bs)
            for t in range(T):
                S = np.zeros((dv, dk))
                for tau in range(t + 1):
                    P = np.eye(dk)
                    for s in range(tau + 1, t + 1):
                        P = P @ A[s]
                    S = S + Bm[tau] @ P
                out[b, hh, t] = S @ q[b, hh, t]
    return out


@pytest.mark.parametrize("L", [1, 2, 4])
def test_brute_force_transition_products(oracle_mod, L):
    inp = f64_inputs(B=1, H=2, T=12, dk=5, dv=4, L=L, seed=7 + L)
    out = run(oracle_mod, inp)["out"]
    ref = _brute_force(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_zero_write_gates_give_zero_state(oracle_mod):
    inp = f64_inputs(B=1, H=2, T=33, dk=6, dv=6, L=3, seed=8)
    inp["beta"] = np.zeros_like(inp["beta"])
    inp["gamma"] = np.zeros_like(inp["gamma"])
    res = run(oracle_mod, inp, want_state=True)
    assert np.all(res["out"] == 0.0) and np.all(res["S_final"] == 0.0)


def test_exact_recall_with_orthonormal_keys(oracle_mod):
    rng = np.random.default_rng(0)
    dk = dv = 16
    T = 16
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qm.T[None, None]                                # rows orthonormal
    v = rng.standard_normal((1, 1, T, dv))
    beta = rng.uniform(0.2, 1.0, (1, 1, T))
    perm = np.array([rng.integers(0, t + 1) for t in range(T)])
    q = k[:, :, perm, :]
    res = oracle_mod.forward(q, k, v, beta, np.ones((1, 1, T)), None, None, None,
                             rng.standard_normal((1, 4, dv)), 1)
    expect = beta[0, 0, perm, None] * v[0, 0, perm]
    np.testing.assert_allclose(res["out"][0, 0], expect, rtol=1e-12, atol=1e-12)
    # beta = 1: plain exact recall o_t = v_{pi(t)}
    res1 = oracle_mod.forward(q, k, v, np.ones((1, 1, T)), np.ones((1, 1, T)), None, None, None,
                              rng.standard_normal((1, 4, dv)), 1)
    np.testing.assert_allclose(res1["out"][0, 0], v[0, 0, perm], rtol=1e-12, atol=1e-12)


def test_no_forget_no_delta_is_causal_linear_attention(oracle_mod):
    inp = f64_inputs(B=1, H=2, T=25, dk=6, dv=5, L=4, seed=9)
    inp["alpha"] = np.ones_like(inp["alpha"])
    inp["beta"] = np.zeros_like(inp["beta"])
    res = run(oracle_mod, inp, want_x=True)
    X, u, q = res["X"], inp["u"], inp["q"]
    T = q.shape[2]
    scores = np.einsum("bhtd,bhjld->bhtjl", q, u)             # q_t . u_{j,l}
    mask = np.tril(np.ones((T, T)))[None, None, :, :, None]
    expect = np.einsum("bhtjl,bhjlc->bhtc", scores * mask, X)
    np.testing.assert_allclose(res["out"], expect, rtol=1e-12, atol=1e-13)


def test_zero_conv_gives_half_gain(oracle_mod):
    inp = f64_inputs(B=1, H=2, T=10, dk=4, dv=4, L=5, seed=10)
    inp["conv_w"] = np.zeros_like(inp["conv_w"])
    res = run(oracle_mod, inp, want_x=True, want_hge=True)
    assert np.all(res["h"] == 0) and np.all(res["g"] == 0.5)
    assert np.array_equal(res["e"], inp["v"])
    v, gam, eta = inp["v"], inp["gamma"], inp["eta"]
    R = inp["L"] - 1
    for l in range(R):
        chain = np.prod(1 - 0.5 * eta[..., :l], axis=-1)      # prod_{j<l}(1 - eta_j / 2)
        expect = gam[..., l, None] * 0.5 * v * chain[..., None]
        np.testing.assert_allclose(res["X"][..., l, :], expect, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("L,dk,dv", [(1, 6, 6), (3, 6, 6), (5, 6, 8), (9, 6, 6)])
def test_single_token_injection_rank(oracle_mod, L, dk, dv):
    inp = f64_inputs(B=1, H=1, T=1, dk=dk, dv=dv, L=L, seed=11 + L)
    res = run(oracle_mod, inp, want_state=True)
    S1 = res["S_final"][0, 0]        # S_0 = 0, so S_1 = B_1
    assert np.linalg.matrix_rank(S1, tol=1e-10) == min(L, dv, dk)


def test_split_call_with_initial_state(oracle_mod):
    """Carrying S_final of a prefix into S_init of the suffix reproduces the full run.
    conv_w = 0 makes the anchor token-local, so no left context is lost at the split."""
    inp = f64_inputs(B=1, H=2, T=30, dk=5, dv=4, L=3, seed=12)
    inp["conv_w"] = np.zeros_like(inp["conv_w"])
    full = run(oracle_mod, inp)
    t0 = 17
    cut = lambda sl: {kk: (vv[:, :, sl] if isinstance(vv, np.ndarray) and kk != "conv_w" else vv)
                      for kk, vv in inp.items()}
    a = run(oracle_mod, cut(slice(0, t0)), want_state=True)
    b = run(oracle_mod, cut(slice(t0, None)), S_init=a["S_final"])
    np.testing.assert_allclose(a["out"], full["out"][:, :, :t0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(b["out"], full["out"][:, :, t0:], rtol=1e-12, atol=1e-13)


def _cut(inp, sl):
    return {kk: (vv[:, :, sl] if isinstance(vv, np.ndarray) and kk != "conv_w" else vv) for kk, vv in inp.items()}


def _history(v_part, prev=None):
    """The three tokens before the next call: v_{-3..-1} from the tokens seen so far (zeros
    before the sequence start)."""
    B, H, _, dv = v_part.shape
    prev = np.zeros((B, H, 3, dv)) if prev is None else prev
    return np.concatenate([prev, v_part], axis=2)[:, :, -3:]


def test_history_equals_prepended_inert_tokens(oracle_mod):
    """v_hist holds v_{-3}, v_{-2}, v_{-1}: a run with it (and an initial state) equals a run on
    the sequence with those three tokens prepended as inert tokens -- alpha = 1 and beta =
    gamma = 0 leave S unchanged whatever their q, k and u -- from the same initial state."""
    inp = f64_inputs(B=1, H=2, T=12, dk=5, dv=4, L=3, seed=16)
    rng = np.random.default_rng(16)
    hist = rng.standard_normal((1, 2, 3, 4))
    S0 = rng.standard_normal((1, 2, 4, 5)) * 0.3
    res = run(oracle_mod, inp, S_init=S0, v_hist=hist, want_state=True)
    pre = {}
    for kk, vv in inp.items():
        if not isinstance(vv, np.ndarray) or kk == "conv_w":
            pre[kk] = vv
            continue
        filler = rng.standard_normal(vv.shape[:2] + (3,) + vv.shape[3:])
        if kk == "v":
            filler = hist
        elif kk == "alpha":
            filler = np.ones_like(filler)
        elif kk in ("beta", "gamma"):
            filler = np.zeros_like(filler)
        pre[kk] = np.concatenate([filler, vv], axis=2)
    ref = run(oracle_mod, pre, S_init=S0, want_state=True)
    np.testing.assert_allclose(res["out"], ref["out"][:, :, 3:], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(res["S_final"], ref["S_final"], rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("cuts", [(17,), (1, 2, 5), (2, 3, 29)])
def test_split_calls_with_history_and_state(oracle_mod, cuts):
    """With a non-zero convolution, consecutive calls that carry S_final into S_init and the
    last three tokens into v_hist reproduce one call over the whole sequence, including calls
    shorter than the convolution window."""
    inp = f64_inputs(B=1, H=2, T=30, dk=5, dv=4, L=3, seed=17)
    assert np.abs(inp["conv_w"]).min() > 0
    full = run(oracle_mod, inp, want_state=True)
    S, hist, outs, t = None, None, [], 0
    for t1 in list(cuts) + [30]:
        part = _cut(inp, slice(t, t1))
        r = run(oracle_mod, part, S_init=S, v_hist=hist, want_state=True)
        outs.append(r["out"])
        S, hist, t = r["S_final"], _history(part["v"], hist), t1
    np.testing.assert_allclose(np.concatenate(outs, axis=2), full["out"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, full["S_final"], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# the non-linear residual variant (notes section 2.3): delta = GELU(p r), r <- r - delta
def nonlinear_inputs(T=20, dk=6, dv=5, L=4, seed=18, p_scale=1.0):
    inp = f64_inputs(B=1, H=2, T=T, dk=dk, dv=dv, L=L, seed=seed)
    rng = np.random.default_rng(seed)
    inp["p_gain"] = p_scale / (1.0 + np.exp(-rng.standard_normal((1, 2, T, L - 1, dv))))
    return inp


def test_nonlinear_zero_gain_is_gdn(oracle_mod):
    """p = 0: GELU(0) = 0, so no level writes and the output is the L = 1 (GDN) output."""
    inp = nonlinear_inputs()
    inp["p_gain"] = np.zeros_like(inp["p_gain"])
    res = run(oracle_mod, inp, p_gain=inp["p_gain"], want_x=True)
    gdn = run(oracle_mod, dict(inp, L=1, u=None, gamma=None, eta=None))
    assert np.all(res["X"] == 0.0)
    np.testing.assert_array_equal(res["out"], gdn["out"])


def test_nonlinear_small_signal_limit_is_the_linear_chain(oracle_mod):
    """GELU(z) = z/2 + O(z^2): for tiny residuals, p = 2 g and eta = 1 turn the non-linear
    chain into the linear one (x_l = gamma g r_l, r_{l+1} = r_l (1 - g)), which the closed-form
    pin above fixes independently."""
    inp = nonlinear_inputs(L=5)
    inp["v"] = inp["v"] * 1e-7
    lin = dict(inp, eta=np.ones_like(inp["eta"]))
    ref = run(oracle_mod, lin, want_x=True, want_hge=True)
    g = ref["g"]
    p = np.repeat(2.0 * g[:, :, :, None, :], 4, axis=3)
    res = run(oracle_mod, inp, p_gain=p, want_x=True)
    scale = np.max(np.abs(ref["X"]))
    assert scale > 0
    assert np.max(np.abs(res["X"] - ref["X"])) <= 1e-5 * scale


def test_nonlinear_saturation_leaves_nothing_for_later_levels(oracle_mod):
    """p = 1 and a large positive residual: GELU(r) = r up to r Phi(-r), so the first level
    takes the whole residual and the later levels see (almost) zero."""
    inp = nonlinear_inputs(L=3)
    inp["v"] = np.full_like(inp["v"], 20.0)
    inp["conv_w"] = np.zeros_like(inp["conv_w"])  # h = 0, so e = v
    p = np.ones_like(inp["p_gain"])
    res = run(oracle_mod, inp, p_gain=p, want_x=True)
    X = res["X"]
    np.testing.assert_allclose(X[:, :, :, 0, :], np.broadcast_to(inp["gamma"][:, :, :, 0, None] * 20.0, X.shape[:3] + X.shape[4:]),
                               rtol=1e-12)
    assert np.max(np.abs(X[:, :, :, 1, :])) < 1e-60


def test_nonlinear_chain_against_library_gelu(oracle_mod):
    """Each level's factor from scipy's normal CDF, level by level, slot l - 1 for level l."""
    inp = nonlinear_inputs(L=4, p_scale=3.0)
    res = run(oracle_mod, inp, p_gain=inp["p_gain"], want_x=True, want_hge=True)
    r = inp["v"] - gelu_lib(res["h"])
    for l in range(3):
        z = inp["p_gain"][:, :, :, l, :] * r
        d = gelu_lib(z)
        np.testing.assert_allclose(res["X"][:, :, :, l, :], inp["gamma"][:, :, :, l, None] * d, rtol=1e-12, atol=1e-15)
        assert d.shape == res["X"][:, :, :, l, :].shape
        r = r - d


def test_state_stays_bounded_long_memory(oracle_mod):
    """beta in (0,1), ||k|| = 1, alpha < 1: the transition is a contraction, so
    ||S_t|| <= max_t ||B_t|| / (1 - max alpha) (notes, section 2.2 stability remark)."""
    inp = f64_inputs(B=1, H=2, T=400, dk=8, dv=8, L=4, seed=13, alpha_div=64.0)
    res = run(oracle_mod, inp, want_state=True, want_x=True)
    v, k, be, u, X = inp["v"], inp["k"], inp["beta"], inp["u"], res["X"]
    bound_B = (be * np.linalg.norm(v, axis=-1) * np.linalg.norm(k, axis=-1)
               + np.sum(np.linalg.norm(X, axis=-1) * np.linalg.norm(u, axis=-1), axis=-1))
    amax = inp["alpha"].max()
    for h in range(2):
        assert np.linalg.norm(res["S_final"][0, h]) <= bound_B[0, h].max() / (1 - amax)
    assert np.all(np.isfinite(res["out"]))


def test_batch_sequences_are_independent(oracle_mod):
    inp = f64_inputs(B=3, H=2, T=20, dk=4, dv=4, L=3, seed=14)
    full = run(oracle_mod, inp)["out"]
    one = {kk: (vv[1:2] if isinstance(vv, np.ndarray) and kk != "conv_w" else vv) for kk, vv in inp.items()}
    np.testing.assert_array_equal(run(oracle_mod, one)["out"][0], full[1])


def test_thread_count_does_not_change_result(oracle_mod):
    inp = f64_inputs(B=2, H=3, T=20, dk=4, dv=4, L=3, seed=15)
    a = run(oracle_mod, inp, nthreads=1)["out"]
    b = run(oracle_mod, inp, nthreads=5)["out"]
    assert np.array_equal(a, b)
