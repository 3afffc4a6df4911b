"""Bounded device waits that run out, on the GPU, with no fault and no hang.

Every wait of the library's TMA / tensor-core pipelines on an mbarrier is bounded by
%globaltimer (PRISM_OPT_WAIT_NS; 100 ms by default).  With the bound set to 1 ns, a wait that
does not find its phase complete gives up at once: the kernel records PRISM_ERR_TIMEOUT in the
plan's status word, waits (bounded by one second) for the copies and products it still has in
flight, frees its tensor memory and returns.  The tests check that the status comes back as
PRISM_ERR_TIMEOUT through prism_plan_last_device_status, that no other error appears, and that
the CUDA context stays usable: with the default bound restored the same plan computes a result
bit-identical to a fresh plan's.  Nothing here faults, traps or spins without a bound.
"""
import pytest
import torch

from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import make_inputs, make_projection_inputs

pytestmark = pytest.mark.gpu

SEQ_KEYS = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")
ATTEMPTS = 16  # a wait that finds its phase already complete does not time out: retry a few times
_FLUSH = {}


def _flush_l2():
    """Write 256 MiB (twice the L2) so that the next call's loads come from HBM and take longer
    than the 1 ns bound."""
    buf = _FLUSH.get("buf")
    if buf is None:
        buf = _FLUSH["buf"] = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    buf.fill_(1.0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _dev(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


def _status(plan):
    """The plan's device status after a sync: PRISM_OK or the PrismError's code (cleared)."""
    torch.cuda.synchronize()
    try:
        plan.last_device_status()
        return B.PRISM_OK
    except B.PrismError as e:
        return e.status


def _expire(plan, run):
    """Run `run` with a 1 ns wait bound until a wait runs out; every other outcome must be OK."""
    plan.set_option(B.PRISM_OPT_WAIT_NS, 1)
    seen = []
    for _ in range(ATTEMPTS):
        _flush_l2()
        run()
        st = _status(plan)
        seen.append(st)
        assert st in (B.PRISM_OK, B.PRISM_ERR_TIMEOUT), seen
        if st == B.PRISM_ERR_TIMEOUT:
            break
    plan.set_option(B.PRISM_OPT_WAIT_NS, 0)  # back to the default bound
    assert B.PRISM_ERR_TIMEOUT in seen, seen
    assert _status(plan) == B.PRISM_OK  # reading the status cleared it


def test_segment_kernel_wait_expires_and_the_plan_recovers():
    """Tensor-core forward: segment kernel (TMA and MMA waits) and combine (bulk-copy ring)."""
    d = _dev(make_inputs(1, 2, 700, 64, 64, 4, dtype="bf16", seed=901))
    with B.Plan.for_inputs(d, path=2, segments=3) as plan:
        _expire(plan, lambda: plan.forward(d))
        again = plan.forward(d)
        assert _status(plan) == B.PRISM_OK
    with B.Plan.for_inputs(d, path=2, segments=3) as fresh:
        ref = fresh.forward(d)
        assert _status(fresh) == B.PRISM_OK
    assert torch.equal(again, ref)


def test_projection_wait_expires_and_the_plan_recovers():
    """Input projections: the TMA ring, the MMA completions and the accumulator hand-over."""
    pi = make_projection_inputs(2, 600, 256, 2, 3, 64, 64, seed=902)
    X, cx, W = pi["X"].cuda(), pi["conv_x"].cuda(), pi["W"].cuda()
    with B.Plan(2, 2, 600, 64, 64, 4, io="bf16") as plan:
        _expire(plan, lambda: plan.project(X, cx, W))
        again = plan.project(X, cx, W)
        assert _status(plan) == B.PRISM_OK
    with B.Plan(2, 2, 600, 64, 64, 4, io="bf16") as fresh:
        ref = fresh.project(X, cx, W)
        assert _status(fresh) == B.PRISM_OK
    for a, b in zip(again, ref):
        assert torch.equal(a, b)


def test_decode_wait_expires_and_the_plan_recovers():
    """Decode step: the producer's and the consumers' waits on the stage ring.  A serving batch
    large enough that every CTA streams many state blocks through its ring, so the producer also
    waits for stages to be released.  The state and history are updated in place, so each call
    gets fresh copies."""
    Bn, H, d = 256, 4, 128
    inp = make_inputs(Bn, H, 1, d, d, 4, dtype="bf16", seed=903)
    dv_ = _dev(inp)
    tok = {k: (v[:, :, 0].contiguous() if k in SEQ_KEYS else v) for k, v in dv_.items()}
    g = torch.Generator().manual_seed(904)
    S0 = (torch.randn(Bn, H, d, d, generator=g) * 0.3).cuda()
    h0 = torch.randn(Bn, H, 3, d, generator=g).to(torch.bfloat16).cuda()
    with B.Plan(Bn, H, 1, d, d, 4, io="bf16") as plan:
        _expire(plan, lambda: plan.decode_step(tok, h0.clone(), S0.clone()))
        S_a, h_a = S0.clone(), h0.clone()
        o_a = plan.decode_step(tok, h_a, S_a)
        assert _status(plan) == B.PRISM_OK
    with B.Plan(Bn, H, 1, d, d, 4, io="bf16") as fresh:
        S_b, h_b = S0.clone(), h0.clone()
        o_b = fresh.decode_step(tok, h_b, S_b)
        assert _status(fresh) == B.PRISM_OK
    assert torch.equal(o_a, o_b) and torch.equal(S_a, S_b) and torch.equal(h_a, h_b)


def test_chunked_backward_wait_expires_and_the_plan_recovers():
    """Chunked backward: the TMA and bulk-copy loads and the product completions of its three
    tensor-core kernels (a few thousand chunk CTAs, so that some product wait is still pending
    when its 1 ns bound is checked)."""
    from ssm_sequence_layer_gb300.inputs import make_cotangents
    d = _dev(make_inputs(2, 4, 8192, 64, 64, 4, dtype="bf16", seed=905))
    dout, _ = make_cotangents(2, 4, 8192, 64, 64, seed=905)
    dout = dout.cuda()
    with B.Plan.for_inputs(d) as plan:
        _expire(plan, lambda: plan.backward(d, dout))
        again = plan.backward(d, dout)
        assert _status(plan) == B.PRISM_OK
    with B.Plan.for_inputs(d) as fresh:
        ref = fresh.backward(d, dout)
        assert _status(fresh) == B.PRISM_OK
    for kk in ref:
        assert torch.equal(again[kk], ref[kk]), kk
