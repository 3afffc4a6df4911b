"""GPU parity of the chunk-map kernels (the tensor-core path for dk = dv = 128, 1 <= L <= 16)
against the fp64 oracle, element by element on the same seeded inputs.

The map kernel turns every 64-token chunk into an affine map of the state entering it
(S -> S A_c + B_c) and of the outputs (O = O_loc + Q~ S^T); the scan kernel applies the maps in
order.  The bar is the bf16 one (2e-2 of max|o - o_ref| / rms(o_ref), fp32 output), as for the
other tensor-core kernels.  The full-size workloads that run on these kernels (the GDN-degenerate
and 130M-LM layer shapes, the 64K-token long-memory case on sampled heads) are in
test_parity_gpu.py.
"""
import numpy as np
import pytest
import torch

from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import make_inputs
from tests.gpu_util import TOL, gpu_forward, oracle_forward, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("B_,H,T,L", [
    (1, 1, 1, 1), (1, 2, 63, 2), (2, 1, 64, 4), (1, 1, 65, 8), (1, 2, 300, 16), (3, 1, 200, 4),
    (1, 1, 1000, 3), (2, 2, 129, 5),
])
def test_map_path_matches_oracle(oracle_mod, B_, H, T, L):
    inp = make_inputs(B_, H, T, 128, 128, L, dtype="bf16", seed=500 + T + L)
    out = gpu_forward(inp, path=2)
    ref = oracle_forward(oracle_mod, inp)["out"]
    err = rel_err(out, ref)
    print(f"B={B_} H={H} T={T} L={L}: rel err {err:.3e}")
    assert np.all(np.isfinite(out))
    assert err <= TOL["bf16"]


def test_map_path_matches_portable_path():
    inp = make_inputs(2, 3, 700, 128, 128, 4, dtype="bf16", seed=520)
    assert rel_err(gpu_forward(inp, path=2), gpu_forward(inp, path=1)) <= TOL["bf16"]


@pytest.mark.parametrize("alpha_div", [1.0, 0.05])
def test_map_path_strong_decay(oracle_mod, alpha_div):
    """About 50 and 1000 nats of decay per chunk."""
    inp = make_inputs(1, 2, 300, 128, 128, 4, dtype="bf16", seed=530, alpha_div=alpha_div)
    out = gpu_forward(inp, path=2)
    ref = oracle_forward(oracle_mod, inp)["out"]
    assert np.all(np.isfinite(out))
    assert rel_err(out, ref) <= TOL["bf16"]


def test_map_path_split_calls_carry_state_and_history(oracle_mod):
    """Calls of 1, 2, 130 and the rest of 300 tokens, each continuing from the previous call's
    final state and convolution history, against one oracle call from the same initial state."""
    inp = make_inputs(2, 2, 300, 128, 128, 4, dtype="bf16", seed=540)
    S0 = torch.randn(2, 2, 128, 128, generator=torch.Generator().manual_seed(541)) * 0.3
    d = to_device(inp)
    S = S0.clone().cuda()
    hist = torch.zeros(2, 2, 3, 128, dtype=torch.bfloat16, device="cuda")
    seq = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta")
    outs, t0 = [], 0
    for t1 in (1, 3, 133, 300):
        part = {k: (v[:, :, t0:t1].contiguous() if k in seq else v) for k, v in d.items()}
        with B.Plan.for_inputs(part, out="f32", path=2) as p:
            outs.append(p.forward_state(part, v_hist=hist, S_init=S, S_final=S, v_hist_out=hist))
            torch.cuda.synchronize()
            p.last_device_status()
        t0 = t1
    ref = oracle_forward(oracle_mod, inp, S_init=S0.double().numpy(), want_state=True)
    assert rel_err(torch.cat(outs, dim=2).double().cpu().numpy(), ref["out"]) <= TOL["bf16"]
    assert rel_err(S.double().cpu().numpy(), ref["S_final"]) <= TOL["bf16"]
    assert torch.equal(hist.cpu(), inp["v"][:, :, -3:])


def test_map_path_bf16_output_is_the_rounded_fp32_output():
    inp = make_inputs(1, 2, 500, 128, 128, 3, dtype="bf16", seed=550)
    d = to_device(inp)
    with B.Plan.for_inputs(d, out="f32", path=2) as p32, B.Plan.for_inputs(d, path=2) as p16:
        o32 = p32.forward(d)
        o16 = p16.forward(d)
        torch.cuda.synchronize()
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_map_path_replays_from_a_cuda_graph():
    inp = make_inputs(1, 2, 400, 128, 128, 4, dtype="bf16", seed=560)
    d = to_device(inp)
    with B.Plan.for_inputs(d, path=2) as p:
        ref = p.forward(d)
        out = torch.zeros_like(ref)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            p.forward(d, out, torch.cuda.current_stream())
        g.replay()
        torch.cuda.synchronize()
        p.last_device_status()
    assert torch.equal(out, ref)


def test_map_path_wait_expires_and_the_plan_recovers():
    """A 1 ns bound on every wait of the map and scan kernels: PRISM_ERR_TIMEOUT comes back, and
    with the default bound the same plan reproduces a fresh plan's output bit for bit.  Sixteen
    sequences of 8192 tokens: a thousand chunks through the map kernel and a hundred and
    twenty-eight ring steps per scan block, so that some wait is still pending when its 1 ns bound
    is checked."""
    d = to_device(make_inputs(2, 8, 8192, 128, 128, 4, dtype="bf16", seed=570))
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    with B.Plan.for_inputs(d, path=2) as plan:
        plan.set_option(B.PRISM_OPT_WAIT_NS, 1)
        seen = []
        for _ in range(16):
            flush.fill_(1.0)
            plan.forward(d)
            torch.cuda.synchronize()
            try:
                plan.last_device_status()
                seen.append(B.PRISM_OK)
            except B.PrismError as e:
                seen.append(e.status)
            assert seen[-1] in (B.PRISM_OK, B.PRISM_ERR_TIMEOUT), seen
            if seen[-1] == B.PRISM_ERR_TIMEOUT:
                break
        assert B.PRISM_ERR_TIMEOUT in seen, seen
        plan.set_option(B.PRISM_OPT_WAIT_NS, 0)
        again = plan.forward(d)
        torch.cuda.synchronize()
        plan.last_device_status()
    with B.Plan.for_inputs(d, path=2) as fresh:
        ref = fresh.forward(d)
        torch.cuda.synchronize()
        fresh.last_device_status()
    assert torch.equal(again, ref)
