"""GPU parity of the state I/O entry points (prism_forward_state, prism_decode_step) against
the fp64 oracle run over the whole sequence in one call.

A sequence is evaluated in consecutive calls that carry the state (fp32) and the last three
v tokens (the anchor's left context) from one call to the next; the concatenated outputs and
the final state must match one oracle call over the whole sequence, at the bars of the
forward: max |o - o_ref| / rms(o_ref) <= 1e-4 for float32 io, 2e-2 for bfloat16 io.  The
state is compared the same way (max |S - S_ref| / rms(S_ref)).
"""
import numpy as np
import pytest
import torch

from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import make_inputs
from tests.gpu_util import TOL, oracle_forward, rel_err, to_device

pytestmark = pytest.mark.gpu

SEQ_KEYS = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def cut(inp, t0, t1):
    return {kk: (vv[:, :, t0:t1].contiguous() if kk in SEQ_KEYS else vv) for kk, vv in inp.items()}


def token(inp, t):
    return {kk: (vv[:, :, t].contiguous() if kk in SEQ_KEYS else vv) for kk, vv in inp.items()}


def init_state(B_, H, dk, dv, seed, scale=0.3):
    g = torch.Generator().manual_seed(seed)
    S = torch.randn(B_, H, dv, dk, generator=g) * scale
    return S


def run_split(inp, cuts, path, S0=None, segments=None):
    """Consecutive prism_forward_state calls over [0, cuts[0]), [cuts[0], cuts[1]), ...; the
    state and the history are updated in place (S_final = S_init, v_hist_out = v_hist)."""
    d = to_device(inp)
    B_, H, T, dk = d["q"].shape
    dv = d["v"].shape[-1]
    S = (S0.clone() if S0 is not None else torch.zeros(B_, H, dv, dk)).cuda().contiguous()
    hist = torch.zeros(B_, H, 3, dv, dtype=d["v"].dtype, device="cuda")
    outs, t0 = [], 0
    for t1 in list(cuts) + [T]:
        part = cut(d, t0, t1)
        kw = dict(path=path) if segments is None else dict(path=path, segments=segments)
        with B.Plan.for_inputs(part, out="f32", **kw) as p:
            outs.append(p.forward_state(part, v_hist=hist, S_init=S, S_final=S, v_hist_out=hist))
            torch.cuda.synchronize()
            p.last_device_status()
        t0 = t1
    return torch.cat(outs, dim=2).double().cpu().numpy(), S.double().cpu().numpy(), hist


# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dt,path,dk,dv,L,cuts,segments", [
    ("f32", 1, 64, 64, 3, (1, 2, 130), None),
    ("f32", 1, 128, 64, 8, (70,), None),
    ("bf16", 1, 64, 128, 2, (2, 65), None),
    ("bf16", 2, 64, 64, 4, (1, 2, 130), None),
    ("bf16", 2, 64, 64, 3, (64, 200), 3),
    ("bf16", 2, 64, 64, 1, (100,), 2),
])
def test_split_calls_match_one_oracle_call(oracle_mod, dt, path, dk, dv, L, cuts, segments):
    inp = make_inputs(2, 2, 300, dk, dv, L, dtype=dt, seed=60 + L + dk)
    S0 = init_state(2, 2, dk, dv, seed=61)
    out, S, hist = run_split(inp, cuts, path, S0=S0, segments=segments)
    ref = oracle_forward(oracle_mod, inp, S_init=S0.double().numpy(), want_state=True)
    assert rel_err(out, ref["out"]) <= TOL[dt]
    assert rel_err(S, ref["S_final"]) <= TOL[dt]
    assert torch.equal(hist.cpu(), inp["v"][:, :, -3:])


@pytest.mark.parametrize("segments", [1, 4])
def test_tensor_core_path_initial_state_and_history(oracle_mod, segments):
    """One call that starts mid-sequence: S_init and v_hist given, S_final asked for, on the
    tensor-core path with one and with several segments."""
    inp = make_inputs(1, 3, 1000, 64, 64, 4, dtype="bf16", seed=62)
    S0 = init_state(1, 3, 64, 64, seed=63)
    hist = torch.randn(1, 3, 3, 64, generator=torch.Generator().manual_seed(64)).to(torch.bfloat16)
    d = to_device(inp)
    S_fin = torch.empty(1, 3, 64, 64, device="cuda")
    with B.Plan.for_inputs(d, out="f32", path=2, segments=segments) as p:
        out = p.forward_state(d, v_hist=hist.cuda(), S_init=S0.cuda(), S_final=S_fin)
        torch.cuda.synchronize()
        p.last_device_status()
    ref = oracle_forward(oracle_mod, inp, S_init=S0.double().numpy(), v_hist=hist.double().numpy(),
                         want_state=True)
    assert rel_err(out.double().cpu().numpy(), ref["out"]) <= TOL["bf16"]
    assert rel_err(S_fin.double().cpu().numpy(), ref["S_final"]) <= TOL["bf16"]


def test_final_state_alone_from_zero(oracle_mod):
    """S_final without S_init (one segment and several) equals the oracle's final state, and the
    outputs are those of prism_forward."""
    inp = make_inputs(2, 1, 700, 64, 64, 3, dtype="bf16", seed=65)
    ref = oracle_forward(oracle_mod, inp, want_state=True)
    d = to_device(inp)
    for path, segments in ((2, 1), (2, 5), (1, None)):
        kw = dict(path=path) if segments is None else dict(path=path, segments=segments)
        S_fin = torch.empty(2, 1, 64, 64, device="cuda")
        with B.Plan.for_inputs(d, out="f32", **kw) as p:
            out = p.forward_state(d, S_final=S_fin)
            plain = p.forward(d)
            torch.cuda.synchronize()
        assert torch.equal(out, plain)
        assert rel_err(S_fin.double().cpu().numpy(), ref["S_final"]) <= TOL["bf16"]


def test_forward_state_without_state_is_prism_forward():
    inp = make_inputs(1, 2, 260, 64, 64, 4, dtype="bf16", seed=66)
    d = to_device(inp)
    for path in (1, 2):
        with B.Plan.for_inputs(d, path=path) as p:
            a = p.forward(d)
            b = p.forward_state(d)
            torch.cuda.synchronize()
        assert torch.equal(a, b)


# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dt,dk,dv,L,prefill", [
    ("bf16", 64, 64, 4, 70),
    ("bf16", 128, 128, 4, 129),
    ("f32", 64, 128, 1, 5),
    ("f32", 128, 64, 8, 2),
    ("bf16", 64, 64, 16, 0),
])
def test_prefill_then_decode_matches_one_oracle_call(oracle_mod, dt, dk, dv, L, prefill):
    """prism_forward_state over the prompt (state and history out), then one prism_decode_step
    per token; every output and the final state against one oracle call over all tokens."""
    T = prefill + 12
    inp = make_inputs(2, 3, T, dk, dv, L, dtype=dt, seed=70 + L + prefill)
    d = to_device(inp)
    S = torch.zeros(2, 3, dv, dk, device="cuda")
    hist = torch.zeros(2, 3, 3, dv, dtype=d["v"].dtype, device="cuda")
    outs = []
    if prefill:
        part = cut(d, 0, prefill)
        with B.Plan.for_inputs(part, out="f32") as p:
            outs.append(p.forward_state(part, S_final=S, v_hist_out=hist))
            torch.cuda.synchronize()
    with B.Plan(2, 3, 1, dk, dv, L, io=dt, out="f32") as p:
        for t in range(prefill, T):
            outs.append(p.decode_step(token(d, t), hist, S).unsqueeze(2))
        torch.cuda.synchronize()
        p.last_device_status()
    ref = oracle_forward(oracle_mod, inp, want_state=True)
    out = torch.cat(outs, dim=2).double().cpu().numpy()
    assert rel_err(out[:, :, prefill:], ref["out"][:, :, prefill:]) <= TOL[dt]
    assert rel_err(out, ref["out"]) <= TOL[dt]
    assert rel_err(S.double().cpu().numpy(), ref["S_final"]) <= TOL[dt]
    assert torch.equal(hist.cpu(), inp["v"][:, :, -3:])


def test_decode_step_equals_one_token_forward():
    """The decode kernel and the chunked portable path with T = 1 compute the same step."""
    inp = make_inputs(3, 2, 1, 128, 64, 5, dtype="f32", seed=80)
    d = to_device(inp)
    S0 = init_state(3, 2, 128, 64, seed=81).cuda()
    h0 = torch.randn(3, 2, 3, 64, generator=torch.Generator().manual_seed(82)).cuda()
    S_a, h_a = S0.clone(), h0.clone()
    S_b = torch.empty_like(S0)
    h_b = torch.empty_like(h0)
    with B.Plan.for_inputs(d, path=1) as p:
        o_a = p.decode_step(token(d, 0), h_a, S_a)
        o_b = p.forward_state(d, v_hist=h0, S_init=S0, S_final=S_b, v_hist_out=h_b)[:, :, 0]
        torch.cuda.synchronize()
    assert rel_err(o_a.cpu().numpy(), o_b.cpu().numpy()) <= 1e-5
    assert rel_err(S_a.cpu().numpy(), S_b.cpu().numpy()) <= 1e-5
    assert torch.equal(h_a, h_b)


def test_decode_steps_replay_from_a_cuda_graph():
    """A serving loop captures the decode step once and replays it: each replay advances the
    state and the history in place exactly as a direct call does."""
    inp = make_inputs(4, 2, 6, 64, 64, 4, dtype="bf16", seed=86)
    d = to_device(inp)
    S0 = init_state(4, 2, 64, 64, seed=87).cuda()
    h0 = torch.zeros(4, 2, 3, 64, dtype=torch.bfloat16, device="cuda")
    with B.Plan(4, 2, 1, 64, 64, 4, io="bf16", out="f32") as p:
        # direct calls on tokens 0..5
        S_a, h_a, outs_a = S0.clone(), h0.clone(), []
        for t in range(6):
            outs_a.append(p.decode_step(token(d, t), h_a, S_a).clone())
        # the same steps from one captured graph: the token's inputs are copied into fixed buffers
        S_b, h_b = S0.clone(), h0.clone()
        tok = {kk: (vv.clone() if torch.is_tensor(vv) else vv) for kk, vv in token(d, 0).items()}
        out = torch.empty(4, 2, 64, device="cuda")
        p.decode_step(tok, h_b.clone(), S_b.clone(), out)  # first call outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            p.decode_step(tok, h_b, S_b, out, torch.cuda.current_stream())
        outs_b = []
        for t in range(6):
            for kk, vv in token(d, t).items():
                if torch.is_tensor(vv) and kk != "conv_w":
                    tok[kk].copy_(vv)
            g.replay()
            outs_b.append(out.clone())
        torch.cuda.synchronize()
        p.last_device_status()
    for a, b in zip(outs_a, outs_b):
        assert torch.equal(a, b)
    assert torch.equal(S_a, S_b) and torch.equal(h_a, h_b)


def test_decode_zero_write_gates_keep_decayed_state():
    """beta = gamma = 0: the step only decays the state, S <- alpha S, and reads it out."""
    inp = make_inputs(2, 2, 1, 64, 64, 3, dtype="f32", seed=83)
    inp["beta"].zero_()
    inp["gamma"].zero_()
    d = to_device(inp)
    S0 = init_state(2, 2, 64, 64, seed=84).cuda()
    S = S0.clone()
    h = torch.zeros(2, 2, 3, 64, device="cuda")
    with B.Plan.for_inputs(d) as p:
        o = p.decode_step(token(d, 0), h, S)
        torch.cuda.synchronize()
    al = d["alpha"][:, :, 0, None, None]
    torch.testing.assert_close(S, al * S0, rtol=1e-6, atol=1e-7)
    torch.testing.assert_close(o, torch.einsum("bhij,bhj->bhi", al * S0, d["q"][:, :, 0]), rtol=1e-5, atol=1e-6)


# ------------------------------------------------------------------------------------------------
def test_state_arguments_are_checked():
    inp = to_device(make_inputs(1, 1, 64, 64, 64, 2, dtype="bf16", seed=85))
    with B.Plan.for_inputs(inp) as p:
        buf = torch.zeros(64 * 64 + 4, device="cuda")
        bad = buf[1:1 + 64 * 64].view(1, 1, 64, 64)  # 4-byte offset
        with pytest.raises(B.PrismError) as ei:
            p.forward_state(inp, S_init=bad)
        assert ei.value.status == B.PRISM_ERR_MISALIGNED
        hist = torch.zeros(1, 1, 3, 64, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(B.PrismError) as ei:
            p.decode_step(token(inp, 0), hist, bad)
        assert ei.value.status == B.PRISM_ERR_MISALIGNED
        with pytest.raises(B.PrismError) as ei:
            B.prism_decode_step(p.handle, *p._tensors(token(inp, 0)), None, bad, hist)
        assert ei.value.status == B.PRISM_ERR_INVALID_ARG


def test_long_sequence_segmented_map_scan(oracle_mod):
    """A sequence of 257 chunks with dk = dv = 128 and two heads: the chunk-map path runs its scan
    as segments (compose, carry, then each segment from its start state).  With S_init given and
    S_final asked for, bf16 output: the whole output and the final state against one oracle call."""
    B_, H, T, L = 1, 2, 257 * 64 - 27, 3
    inp = make_inputs(B_, H, T, 128, 128, L, dtype="bf16", seed=71)
    S0 = init_state(B_, H, 128, 128, seed=72)
    d = to_device(inp)
    S_fin = torch.empty(B_, H, 128, 128, device="cuda")
    with B.Plan.for_inputs(d, out="f32") as p:
        out = p.forward_state(d, S_init=S0.cuda(), S_final=S_fin)
        torch.cuda.synchronize()
        p.last_device_status()
    ref = oracle_forward(oracle_mod, inp, S_init=S0.double().numpy(), want_state=True)
    got = out.double().cpu().numpy()
    err_o, err_s = rel_err(got, ref["out"]), rel_err(S_fin.double().cpu().numpy(), ref["S_final"])
    print(f"segmented map scan: rel err out {err_o:.3e}, S_final {err_s:.3e}")
    assert np.all(np.isfinite(got))
    assert err_o <= TOL["bf16"] and err_s <= TOL["bf16"]
