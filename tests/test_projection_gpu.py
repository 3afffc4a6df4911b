"""GPU parity of the block's input projections (prism_project) against the fp64 oracle
(oracle/prism_projection.py) on the same bf16 inputs.  Bars: max |x - x_ref| / rms(x_ref) <= 2e-2
for the basis and gain outputs (bf16 operands and outputs, fp32 accumulation); max |gamma -
gamma_ref| <= 5e-3 for the gates, derived from the arithmetic: the anchor enters the tensor
cores rounded to bf16 (relative 2^-9 per entry), which moves a logit z by up to about
2^-9 |z| with |z| <= ~8 on these inputs, and the logistic's slope is at most 1/4."""
import numpy as np
import pytest
import torch

from oracle import prism_projection as PP
from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import make_gain, make_inputs, make_projection_inputs
from tests.gpu_util import TOL, oracle_forward, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def run_project(pi, L=None):
    B_, T, D, H, R, dk, dv = (pi[k] for k in ("B", "T", "D", "H", "R", "dk", "dv"))
    with B.Plan(B_, H, T, dk, dv, R + 1, io="bf16") as plan:
        u, p, g = plan.project(pi["X"].cuda(), pi["conv_x"].cuda(), pi["W"].cuda())
        torch.cuda.synchronize()
        plan.last_device_status()
    return u, p, g


@pytest.mark.parametrize("B_,T,D,H,R,dk,dv", [
    (2, 300, 128, 2, 2, 64, 64),
    (1, 129, 256, 2, 3, 128, 64),
    (1, 1, 64, 1, 1, 64, 64),
    (3, 130, 192, 1, 1, 64, 128),
    (1, 512, 512, 4, 3, 128, 128),
])
def test_projection_matches_oracle(B_, T, D, H, R, dk, dv):
    pi = make_projection_inputs(B_, T, D, H, R, dk, dv, seed=T + D)
    u, p, g = run_project(pi)
    ru, rp, rg = PP.project(pi["X"], pi["conv_x"], pi["W"], H, R, dk, dv)
    assert rel_err(u.double().cpu().numpy(), ru) <= TOL["bf16"]
    assert rel_err(p.double().cpu().numpy(), rp) <= TOL["bf16"]
    assert np.max(np.abs(g.double().cpu().numpy() - rg)) <= 5e-3
    un = torch.linalg.vector_norm(u.float(), dim=-1)
    assert torch.all((un - 1).abs() < 1e-2)


def test_projection_feeds_the_nonlinear_variant(oracle_mod):
    """The projections' outputs are the recurrence's directions, gains and gates: projecting and
    running prism_forward_nonlinear matches the two oracles chained."""
    B_, T, D, H, R, d = 1, 200, 128, 2, 3, 64
    pi = make_projection_inputs(B_, T, D, H, R, d, d, seed=5)
    u, p, g = run_project(pi)
    inp = make_inputs(B_, H, T, d, d, R + 1, dtype="bf16", seed=6)
    inp.update(u=u.cpu(), gamma=g.cpu())
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    with B.Plan.for_inputs(dev, out="f32") as plan:
        out = plan.forward_nonlinear(dev, p).double().cpu().numpy()
        torch.cuda.synchronize()
    ref = oracle_forward(oracle_mod, inp, p_gain=p.double().cpu().numpy())["out"]
    assert rel_err(out, ref) <= TOL["bf16"]


def test_projection_argument_errors():
    pi = make_projection_inputs(1, 64, 96, 1, 1, 64, 64, seed=1)
    with B.Plan(1, 1, 64, 64, 64, 2, io="bf16") as plan:
        with pytest.raises(B.PrismError) as ei:
            plan.project(pi["X"].cuda(), pi["conv_x"].cuda(), torch.zeros(129, 96, dtype=torch.bfloat16).cuda())
        assert ei.value.status == B.PRISM_ERR_UNSUPPORTED
    with B.Plan(1, 1, 64, 64, 64, 2, io="f32") as plan:
        with pytest.raises(B.PrismError) as ei:
            plan.project(torch.zeros(1, 64, 64, dtype=torch.bfloat16).cuda(), torch.zeros(4, 64, dtype=torch.bfloat16).cuda(),
                         torch.zeros(129, 64, dtype=torch.bfloat16).cuda())
        assert ei.value.status == B.PRISM_ERR_UNSUPPORTED
