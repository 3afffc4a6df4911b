"""GPU parity of prism_backward's chunked tensor-core form (bf16 io, dk = dv = 64, 1 <= L <= 4, the
form the automatic path takes for those shapes) against the fp64 backward oracle.

The chunk-level arrangement (per-chunk maps, a scan of the chunk-boundary states and cotangents,
per-chunk cotangent products) is exact algebra, checked in fp64 by test_backward_chunk_maps.py; the
GPU adds rounding only.  Its products take fp16 operands (unit roundoff 2^-11) with fp32
accumulation over at most 256 terms, and each cotangent passes through at most three dependent
rounded products (e.g. dq <- J <- z <- Wbar), so the bar is max |g - g_ref| / rms(g_ref) <= 1e-2 per
cotangent tensor: ten times the ~1e-3 that three roundings of 2^-11 amplified by sqrt(64)-sized
sums give, and below the forward's bf16 bar of 2e-2.  A dropped or mis-signed term moves a
cotangent by O(rms), far above it.
"""
import numpy as np
import pytest
import torch

from oracle import prism_backward
from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import WORKLOADS, make_cotangents, make_inputs, make_workload_inputs
from tests.gpu_util import rel_err, to_device

pytestmark = pytest.mark.gpu

TC_BAR = 1e-2
PER_HEAD = ("dq", "dk", "dv", "dbeta", "dalpha", "du", "dgamma", "deta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def side_inputs(B_, H, d, seed):
    g = torch.Generator().manual_seed(seed + 31)
    S0 = torch.randn(B_, H, d, d, generator=g) * 0.3
    vh = torch.randn(B_, H, 3, d, generator=g).to(torch.bfloat16)
    return S0, vh


def gpu_backward(inp, dout, dS_final=None, v_hist=None, S_init=None, path=None):
    d = to_device(inp)
    with B.Plan.for_inputs(d, path=path) as p:
        g = p.backward(d, dout.cuda(), dS_final=None if dS_final is None else dS_final.cuda(),
                       v_hist=None if v_hist is None else v_hist.cuda(),
                       S_init=None if S_init is None else S_init.cuda(), want_dv_hist=True, want_dS_init=True)
        torch.cuda.synchronize()
        p.last_device_status()
        ws = p.workspace_bytes()
    return {kk: vv.double().cpu().numpy() for kk, vv in g.items()}, ws


def oracle_backward(inp, dout, dS_final=None, v_hist=None, S_init=None):
    return prism_backward.backward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"], inp["gamma"],
                                   inp["eta"], inp["conv_w"], inp["L"], dout, S_init=S_init, v_hist=v_hist,
                                   dS_final=dS_final, want_dv_hist=True, want_dS_init=True)


def compare(got, ref, keys, bar=TC_BAR):
    errs = {kk: rel_err(got[kk], ref[kk]) for kk in keys if ref[kk].size}
    print("chunked backward parity: " + ", ".join(f"{kk} {e:.2e}" for kk, e in errs.items()))
    bad = {kk: e for kk, e in errs.items() if not e <= bar}
    assert not bad, f"cotangents over the bar {bar}: {bad} (all: {errs})"
    return errs


CASES = [
    # B, H, T, L, state (S_init, v_hist, dS_final)
    (1, 2, 200, 3, True),
    (2, 1, 130, 4, True),
    (1, 2, 97, 1, False),
    (1, 1, 64, 2, True),
    (2, 2, 300, 4, False),
    (1, 1, 1, 4, True),
    (1, 1, 5, 3, True),
    (1, 3, 129, 4, True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}T{c[2]}L{c[3]}{'-state' if c[4] else ''}" for c in CASES])
def test_chunked_backward_matches_oracle(case):
    B_, H, T, L, state = case
    inp = make_inputs(B_, H, T, 64, 64, L, dtype="bf16", seed=T + 7 * L)
    dout, dS_final = make_cotangents(B_, H, T, 64, 64, seed=T + 7 * L, with_state=state)
    S0, vh = side_inputs(B_, H, 64, T) if state else (None, None)
    got, _ = gpu_backward(inp, dout, dS_final, vh, S0)
    ref = oracle_backward(inp, dout, dS_final, vh, S0)
    keys = list(PER_HEAD) + ["dconv_w", "dv_hist", "dS_init"]
    if L == 1:
        keys = [kk for kk in keys if kk not in ("du", "dgamma", "deta")]
        assert np.all(got["dconv_w"] == 0.0)
    compare(got, ref, keys)


def test_unread_gain_slot_is_never_read():
    """NaN in eta[..., R-1] (a gain the forward never reads) leaves every cotangent finite."""
    inp = make_inputs(1, 2, 150, 64, 64, 4, dtype="bf16", seed=12)
    inp["eta"][..., -1] = float("nan")
    dout, dS_final = make_cotangents(1, 2, 150, 64, 64, seed=12, with_state=True)
    got, _ = gpu_backward(inp, dout, dS_final)
    for kk, vv in got.items():
        assert np.all(np.isfinite(vv)), kk
    compare(got, oracle_backward(inp, dout, dS_final), list(PER_HEAD) + ["dconv_w", "dv_hist", "dS_init"])


def test_chunked_backward_is_deterministic():
    inp = make_inputs(2, 2, 300, 64, 64, 4, dtype="bf16", seed=9)
    dout, dS_final = make_cotangents(2, 2, 300, 64, 64, seed=9, with_state=True)
    a, _ = gpu_backward(inp, dout, dS_final)
    b, _ = gpu_backward(inp, dout, dS_final)
    for kk in a:
        assert np.array_equal(a[kk], b[kk]), kk


@pytest.mark.parametrize("name", ["seqrec_16k"])
def test_full_size_sampled_sequences(name):
    """The whole 16K-token workload in one call (the configuration bench.py --mode backward times);
    two of its sequences through the oracle.  The workspace holds per-chunk maps and states, not
    per-token ones: well under the 2 B H T dv dk floats of the token-serial form."""
    w = WORKLOADS[name]
    inp = make_workload_inputs(w, seed=0)
    dout, _ = make_cotangents(w.B, w.H, w.T, w.dk, w.dv, seed=0)
    got, ws = gpu_backward(inp, dout)
    assert ws < 2 * w.B * w.H * w.T * w.dv * w.dk * 4 / 4, ws
    for b, h in [(0, 1), (w.B - 1, w.H - 1)]:
        one = {kk: (vv[b:b + 1, h:h + 1].contiguous() if kk not in ("L", "conv_w") else vv) for kk, vv in inp.items()}
        one["conv_w"] = inp["conv_w"][h:h + 1].contiguous()
        ref = oracle_backward(one, dout[b:b + 1, h:h + 1])
        mine = {kk: got[kk][b:b + 1, h:h + 1] for kk in PER_HEAD}
        compare(mine, ref, PER_HEAD)


def test_portable_and_chunked_forms_agree():
    """The same plan shape through both forms (PRISM_OPT_PATH = 1 forces the token-serial one)."""
    inp = make_inputs(1, 2, 257, 64, 64, 4, dtype="bf16", seed=21)
    dout, dS_final = make_cotangents(1, 2, 257, 64, 64, seed=21, with_state=True)
    tc, ws_tc = gpu_backward(inp, dout, dS_final)
    ts, ws_ts = gpu_backward(inp, dout, dS_final, path=1)
    assert ws_tc != ws_ts
    compare(tc, ts, list(PER_HEAD) + ["dconv_w", "dv_hist", "dS_init"])


@pytest.mark.parametrize("alpha_div", [4.0, 1.0, 0.25])
def test_chunked_backward_under_strong_decay(alpha_div):
    """Gates alpha = exp(-softplus(N(0, 1)) / alpha_div) below the workloads' (alpha_div = 4: alpha
    from ~0.3; 1: median ~0.5; 0.25: median ~0.06, a chunk decaying by e^-200 and more): the pair
    decays underflow inside a chunk and every cotangent but dalpha meets the bar.  dalpha comes from
    alpha_t dalpha_t = <G, S'> + a suffix sum of per-token terms of order one that cancels down to
    order alpha_t, so its rounding error grows like 1 / alpha_t; it meets the bar on the tokens
    with alpha_t >= 0.5 (the workloads' gates are >= 0.73)."""
    inp = make_inputs(1, 2, 300, 64, 64, 4, dtype="bf16", seed=44, alpha_div=alpha_div)
    dout, dS_final = make_cotangents(1, 2, 300, 64, 64, seed=44, with_state=True)
    S0, vh = side_inputs(1, 2, 64, 300)
    got, _ = gpu_backward(inp, dout, dS_final, vh, S0)
    ref = oracle_backward(inp, dout, dS_final, vh, S0)
    for kk, vv in got.items():
        assert np.all(np.isfinite(vv)), kk
    keys = [kk for kk in list(PER_HEAD) + ["dconv_w", "dv_hist", "dS_init"] if kk != "dalpha"]
    compare(got, ref, keys)
    alpha = inp["alpha"].double().numpy()
    for lo in (0.9, 0.5, 0.25, 0.1, 0.0):
        sel = alpha >= lo
        if sel.any():
            print(f"dalpha on alpha >= {lo}: {sel.mean():.2f} of tokens, err {rel_err(got['dalpha'][sel], ref['dalpha'][sel]):.2e}")
    sel = alpha >= 0.5
    if sel.any():
        e = rel_err(got["dalpha"][sel], ref["dalpha"][sel])
        assert e <= TC_BAR, e
