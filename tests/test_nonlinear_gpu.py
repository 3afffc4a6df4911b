"""GPU parity of the non-linear residual variant (prism_forward_nonlinear) against the fp64
oracle with the same gains: delta = GELU(p r), r <- r - delta (notes on PRISM, section 2.3).
Bars as for the forward: max |o - o_ref| / rms(o_ref) <= 1e-4 for float32 io, 2e-2 for
bfloat16 io (fp32 output compared)."""
import numpy as np
import pytest
import torch

from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import make_gain, make_inputs
from tests.gpu_util import TOL, oracle_forward, rel_err, to_device

pytestmark = pytest.mark.gpu
SEQ_KEYS = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_nl(inp, p, **kw):
    d = to_device(inp)
    with B.Plan.for_inputs(d, out="f32") as plan:
        out = plan.forward_nonlinear(d, p.cuda(), **kw)
        torch.cuda.synchronize()
        plan.last_device_status()
    return out.double().cpu().numpy()


@pytest.mark.parametrize("B_,H,T,dk,dv,L,dt", [
    (1, 2, 200, 64, 64, 3, "f32"),
    (2, 1, 65, 128, 64, 8, "f32"),
    (1, 2, 300, 64, 64, 4, "bf16"),
    (2, 2, 257, 128, 128, 4, "bf16"),
    (1, 1, 1, 64, 128, 16, "bf16"),
])
def test_nonlinear_variant_matches_oracle(oracle_mod, B_, H, T, dk, dv, L, dt):
    inp = make_inputs(B_, H, T, dk, dv, L, dtype=dt, seed=90 + L + T)
    p = make_gain(B_, H, T, L, dv, dtype=dt, seed=90 + L + T)
    out = run_nl(inp, p)
    ref = oracle_forward(oracle_mod, inp, p_gain=p.double().numpy())["out"]
    assert rel_err(out, ref) <= TOL[dt]


def test_nonlinear_variant_differs_from_linear_chain(oracle_mod):
    """The variant is a different computation: its output is far from prism_forward's."""
    inp = make_inputs(1, 2, 200, 64, 64, 4, dtype="f32", seed=95)
    p = make_gain(1, 2, 200, 4, 64, dtype="f32", seed=95)
    d = to_device(inp)
    with B.Plan.for_inputs(d, out="f32") as plan:
        lin = plan.forward(d).cpu().numpy()
    nl = run_nl(inp, p)
    assert rel_err(nl, lin) > 1e-2


def test_nonlinear_zero_gain_is_gdn():
    inp = make_inputs(1, 2, 150, 64, 64, 3, dtype="f32", seed=96)
    p = torch.zeros(1, 2, 150, 2, 64)
    nl = run_nl(inp, p)
    gdn_inp = dict(inp, L=1)
    d = to_device(gdn_inp)
    with B.Plan.for_inputs(d, out="f32") as plan:
        gdn = plan.forward(d).double().cpu().numpy()
    assert rel_err(nl, gdn) <= 1e-6


def test_nonlinear_split_calls_with_state(oracle_mod):
    """Consecutive calls carrying the state and the convolution history reproduce one oracle
    call over the whole sequence."""
    inp = make_inputs(1, 2, 230, 64, 64, 4, dtype="f32", seed=97)
    p = make_gain(1, 2, 230, 4, 64, dtype="f32", seed=97)
    d = to_device(inp)
    S = torch.zeros(1, 2, 64, 64, device="cuda")
    hist = torch.zeros(1, 2, 3, 64, device="cuda")
    outs, t0 = [], 0
    for t1 in (2, 100, 230):
        part = {kk: (vv[:, :, t0:t1].contiguous() if kk in SEQ_KEYS else vv) for kk, vv in d.items()}
        with B.Plan.for_inputs(part, out="f32") as plan:
            outs.append(plan.forward_nonlinear(part, p[:, :, t0:t1].contiguous().cuda(), v_hist=hist, S_init=S,
                                               S_final=S, v_hist_out=hist))
            torch.cuda.synchronize()
        t0 = t1
    ref = oracle_forward(oracle_mod, inp, p_gain=p.double().numpy(), want_state=True)
    assert rel_err(torch.cat(outs, dim=2).double().cpu().numpy(), ref["out"]) <= TOL["f32"]
    assert rel_err(S.double().cpu().numpy(), ref["S_final"]) <= TOL["f32"]


@pytest.mark.parametrize("B_,H,T,d,L", [
    (1, 2, 300, 64, 4), (2, 1, 1000, 64, 3), (1, 1, 65, 64, 2),       # segment kernels
    (2, 2, 257, 128, 4), (1, 1, 130, 128, 8), (1, 2, 64, 128, 16),    # chunk-map kernels
])
def test_nonlinear_variant_on_the_tensor_core_path(oracle_mod, B_, H, T, d, L):
    """The variant on the tensor-core kernels (forced, and chosen automatically for bf16): only
    their prep differs, stepping delta = GELU(p r), r <- r - delta level by level."""
    inp = make_inputs(B_, H, T, d, d, L, dtype="bf16", seed=110 + L + T)
    p = make_gain(B_, H, T, L, d, dtype="bf16", seed=110 + L + T)
    ref = oracle_forward(oracle_mod, inp, p_gain=p.double().numpy())["out"]
    dd = to_device(inp)
    for kw in (dict(path=2), {}):
        with B.Plan.for_inputs(dd, out="f32", **kw) as plan:
            out = plan.forward_nonlinear(dd, p.cuda())
            torch.cuda.synchronize()
            plan.last_device_status()
        assert rel_err(out.double().cpu().numpy(), ref) <= TOL["bf16"]


def test_nonlinear_variant_checks_its_gains():
    inp = to_device(make_inputs(1, 1, 64, 64, 64, 3, dtype="bf16", seed=98))
    with B.Plan.for_inputs(inp) as plan:
        with pytest.raises(B.PrismError) as ei:
            B.prism_forward_nonlinear(plan.handle, *plan._tensors(inp)[:7], None, inp["conv_w"], 3, None, None,
                                      torch.empty_like(inp["v"]), None, None)
        assert ei.value.status == B.PRISM_ERR_INVALID_ARG
