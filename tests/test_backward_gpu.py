"""GPU parity of prism_backward's token-serial form (PRISM_OPT_PATH = 1, every shape) against the
fp64 backward oracle on the same seeded inputs.

The token-serial form computes in fp32 from the io values, which the oracle receives exactly (bf16
inputs are widened to fp64).  So no bf16 rounding happens inside, and the bars are those of
fp32 arithmetic: max |g - g_ref| / rms(g_ref) <= 1e-4 per cotangent tensor for float32 io (the
forward's own fp32 bar) and <= 1e-3 for bfloat16 io, whose workloads here run 16K-token chains.
Small cases span several 64-token tiles of the convolution kernel and a ragged tail; the
full-size recommendation shape is compared on sampled (batch, head) sequences, which the
oracle computes one by one (the convolution weight's cotangent sums over the batch, so it is
compared at the small sizes only).
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

BAR = {"f32": 1e-4, "bf16": 1e-3}
PER_HEAD = ("dq", "dk", "dv", "dbeta", "dalpha", "du", "dgamma", "deta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def side_inputs(B_, H, dk, dv, seed, io):
    g = torch.Generator().manual_seed(seed + 31)
    S0 = torch.randn(B_, H, dv, dk, generator=g) * 0.3
    vh = torch.randn(B_, H, 3, dv, generator=g).to(torch.bfloat16 if io == "bf16" else torch.float32)
    return S0, vh


def gpu_backward(inp, dout, dS_final=None, v_hist=None, S_init=None, path=1):
    d = to_device(inp)
    with B.Plan.for_inputs(d, path=path) as p:
        g = p.backward(d, dout.cuda(), dS_final=None if dS_final is None else dS_final.cuda(),
                       v_hist=None if v_hist is None else v_hist.cuda(),
                       S_init=None if S_init is None else S_init.cuda(), want_dv_hist=True, want_dS_init=True)
        torch.cuda.synchronize()
        p.last_device_status()
    return {kk: vv.double().cpu().numpy() for kk, vv in g.items()}


def oracle_backward(inp, dout, dS_final=None, v_hist=None, S_init=None):
    return prism_backward.backward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"], inp["gamma"],
                                   inp["eta"], inp["conv_w"], inp["L"], dout, S_init=S_init, v_hist=v_hist,
                                   dS_final=dS_final, want_dv_hist=True, want_dS_init=True)


def compare(got, ref, io, keys):
    errs = {kk: rel_err(got[kk], ref[kk]) for kk in keys if ref[kk].size}
    print(f"backward parity ({io}): " + ", ".join(f"{kk} {e:.2e}" for kk, e in errs.items()))
    bad = {kk: e for kk, e in errs.items() if not e <= BAR[io]}
    assert not bad, f"cotangents over the bar {BAR[io]}: {bad} (all: {errs})"
    return errs


CASES = [
    # B, H, T, dk, dv, L, io, state
    (1, 2, 200, 64, 64, 3, "f32", True),
    (2, 1, 130, 128, 128, 4, "bf16", True),
    (1, 2, 97, 64, 64, 1, "bf16", False),
    (1, 1, 77, 64, 128, 2, "f32", True),
    (1, 1, 70, 128, 64, 5, "bf16", False),
    (1, 1, 40, 64, 64, 16, "f32", True),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}T{c[2]}dk{c[3]}dv{c[4]}L{c[5]}{c[6]}"
                                             f"{'-state' if c[7] else ''}" for c in CASES])
def test_backward_matches_oracle(case):
    B_, H, T, dk, dv, L, io, state = case
    inp = make_inputs(B_, H, T, dk, dv, L, dtype=io, seed=T + L)
    dout, dS_final = make_cotangents(B_, H, T, dk, dv, seed=T + L, with_state=state)
    S0, vh = side_inputs(B_, H, dk, dv, T, io) if state else (None, None)
    got = gpu_backward(inp, dout, dS_final, vh, S0)
    ref = oracle_backward(inp, dout, dS_final, vh, S0)
    keys = list(PER_HEAD) + ["dconv_w", "dv_hist", "dS_init"]
    if L == 1:
        keys = [kk for kk in keys if kk not in ("du", "dgamma", "deta")]
        assert np.all(got["dconv_w"] == 0.0)
    compare(got, ref, io, keys)


@pytest.mark.parametrize("T", [1, 2, 3, 5])
def test_short_sequences_with_history(T):
    """Sequences shorter than the convolution window: every token reads the history."""
    inp = make_inputs(1, 2, T, 64, 64, 3, dtype="f32", seed=50 + T)
    dout, dS_final = make_cotangents(1, 2, T, 64, 64, seed=50 + T, with_state=True)
    S0, vh = side_inputs(1, 2, 64, 64, T, "f32")
    got = gpu_backward(inp, dout, dS_final, vh, S0)
    ref = oracle_backward(inp, dout, dS_final, vh, S0)
    compare(got, ref, "f32", list(PER_HEAD) + ["dconv_w", "dv_hist", "dS_init"])


def test_unread_gain_slot_is_never_read():
    """NaN in eta[..., R-1] (a gain the forward never reads) leaves every cotangent finite and
    equal to the oracle's."""
    inp = make_inputs(1, 2, 150, 64, 64, 4, dtype="bf16", seed=12)
    inp["eta"][..., -1] = float("nan")
    dout, dS_final = make_cotangents(1, 2, 150, 64, 64, seed=12, with_state=True)
    got = gpu_backward(inp, dout, dS_final)
    ref = oracle_backward(inp, dout, dS_final)
    for kk, vv in got.items():
        assert np.all(np.isfinite(vv)), kk
    compare(got, ref, "bf16", list(PER_HEAD) + ["dconv_w", "dv_hist", "dS_init"])


def test_backward_is_deterministic():
    inp = make_inputs(2, 2, 300, 64, 64, 4, dtype="bf16", seed=9)
    dout, dS_final = make_cotangents(2, 2, 300, 64, 64, seed=9, with_state=True)
    a = gpu_backward(inp, dout, dS_final)
    b = gpu_backward(inp, dout, dS_final)
    for kk in a:
        assert np.array_equal(a[kk], b[kk]), kk


def test_backward_reuses_its_workspace_and_rejects_bad_arguments():
    inp = make_inputs(1, 2, 64, 64, 64, 3, dtype="bf16", seed=4)
    d = to_device(inp)
    dout, _ = make_cotangents(1, 2, 64, 64, 64, seed=4)
    with B.Plan.for_inputs(d, path=1) as p:
        g1 = p.backward(d, dout.cuda())
        ws = p.workspace_bytes()
        g2 = p.backward(d, dout.cuda())
        torch.cuda.synchronize()
        assert p.workspace_bytes() == ws
        assert torch.equal(g1["dq"], g2["dq"])
        with pytest.raises(B.PrismError):
            B.prism_backward(p.handle, d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["u"], d["gamma"], d["eta"],
                             d["conv_w"], 3, None, None, dout.cuda(), None, g1["dq"], g1["dk"], g1["dv"], g1["dbeta"],
                             g1["dalpha"], None, g1["dgamma"], g1["deta"], g1["dconv_w"], None, None)
        with pytest.raises(B.PrismError):
            B.prism_backward(p.handle, d["q"], d["k"], d["v"], d["beta"], d["alpha"], d["u"], d["gamma"], d["eta"],
                             d["conv_w"], 2, None, None, dout.cuda(), None, g1["dq"], g1["dk"], g1["dv"], g1["dbeta"],
                             g1["dalpha"], g1["du"], g1["dgamma"], g1["deta"], g1["dconv_w"], None, None)


@pytest.mark.parametrize("name", ["seqrec_16k", "long_64k"])
def test_full_size_sampled_sequences(name):
    """The whole workload on the GPU in one call; two of its sequences through the oracle.  The
    64K-token stress shape (16 heads of 128, L = 8) is the largest: its per-token states and
    cotangents take 2 B H T dv dk 4 bytes = 137 GB of the device's memory."""
    w = WORKLOADS[name]
    inp = make_workload_inputs(w, seed=0)
    dout, _ = make_cotangents(w.B, w.H, w.T, w.dk, w.dv, seed=0)
    pairs = [(0, 1), (w.B - 1, w.H - 1)]
    d = to_device(inp)
    with B.Plan.for_inputs(d, path=1) as p:
        g = p.backward(d, dout.cuda())
        torch.cuda.synchronize()
        p.last_device_status()
        got = {kk: [vv[b:b + 1, h:h + 1].double().cpu().numpy() for b, h in pairs] for kk, vv in g.items()
               if kk in PER_HEAD}
    del d, g
    torch.cuda.empty_cache()
    for n_, (b, h) in enumerate(pairs):
        one = {kk: (vv[b:b + 1, h:h + 1].contiguous() if kk not in ("L", "conv_w") else vv) for kk, vv in inp.items()}
        one["conv_w"] = inp["conv_w"][h:h + 1].contiguous()
        ref = oracle_backward(one, dout[b:b + 1, h:h + 1])
        mine = {kk: got[kk][n_] for kk in PER_HEAD}
        compare(mine, ref, w.dtype, PER_HEAD)
