"""prism_forward_noalloc: the forward for callers that cannot allocate device memory while
they run -- code inside a device-memory allocator or pool hook (a nested cudaMalloc would
recurse or deadlock), real-time loops whose memory is reserved up front, hosts that forbid
allocation after start-up.  Its scratch is a fixed array compiled into the library, shared
by every call.

The test calls it twice in a row through the C ABI, on two different input sets, and
compares each output with the plan-based prism_forward: a default plan picks the same
tensor-core path and the same automatic segment count, so the two run the same kernels on the
same segmentation and must agree bit for bit.  The second call also shows that the scratch left
over by the first call does not leak into the next result.  The first output is also checked
against the fp64 oracle.  This file is named to be collected last.
"""
import pytest
import torch

from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import make_inputs
from tests.gpu_util import TOL, oracle_forward, rel_err_bf16_out, to_device

pytestmark = pytest.mark.gpu


def test_noalloc_matches_plan_forward_on_two_calls_in_a_row(oracle_mod):
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    Bn, H, T, d, L = 2, 4, 1500, 64, 4            # 24 chunks with a ragged tail, several segments
    stream = torch.cuda.current_stream()
    for seed in (50, 51):
        cpu = make_inputs(Bn, H, T, d, d, L, dtype="bf16", seed=seed)
        inp = to_device(cpu)
        with B.Plan.for_inputs(inp) as plan:     # automatic path and segment count, bf16 output
            ref = plan.forward(inp, stream=stream)
            torch.cuda.synchronize()
            plan.last_device_status()
        out = torch.full_like(inp["v"], float("nan"))
        status = B.prism_forward_noalloc(Bn, H, T, d, d, L, inp["q"], inp["k"], inp["v"], inp["beta"],
                                         inp["alpha"], inp["u"], inp["gamma"], inp["eta"], inp["conv_w"], out,
                                         stream=stream)
        torch.cuda.synchronize()
        assert status == 0
        assert torch.equal(out, ref)
        if seed == 50:
            err = rel_err_bf16_out(out.double().cpu().numpy(), oracle_forward(oracle_mod, cpu)["out"])
            assert err <= TOL["bf16"], err


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build.build()
    lib = B.lib()
    # 64 MiB holds neither the per-chunk stash of 2048 sequences x 64K tokens nor their maps alone
    rc = lib.prism_forward_noalloc(64, 32, 65536, 64, 64, 4, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, None, None)
    assert rc == B.PRISM_ERR_UNSUPPORTED
    assert "too large for the fixed scratch" in B.prism_last_error_message()
    rc = lib.prism_forward_noalloc(1, 1, 64, 128, 128, 2, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, None, None)
    assert rc == B.PRISM_ERR_UNSUPPORTED
