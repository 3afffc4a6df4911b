"""prism_forward_noalloc: the forward for callers that cannot allocate device memory while
they run -- code inside a device-memory allocator or pool hook (a nested cudaMalloc would
recurse or deadlock), real-time loops whose memory is reserved up front, hosts that forbid
allocation after start-up.  Its scratch is a fixed array compiled into the library, shared
by every call.

The test calls it twice in a row through the C ABI, on two different input sets, and
compares each output with the plan-based prism_forward on the same tensor-core path and
segment count, within the bar the parity tests use.  The second call also shows that the
scratch left over by the first call does not leak into the next result.  This file is
named to be collected last.
"""
import ctypes

import pytest
import torch

from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build
from ssm_sequence_layer_gb300.inputs import make_inputs
from tests.gpu_util import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


def test_noalloc_matches_plan_forward_on_two_calls_in_a_row():
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    Bn, H, T, d, L = 2, 4, 1500, 64, 4            # 24 chunks with a ragged tail
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    NC = -(-T // 64)
    P = min(NC, max(1, sms // (Bn * H)))         # the segment count the call chooses here
    stream = torch.cuda.current_stream()
    for seed in (50, 51):
        inp = to_device(make_inputs(Bn, H, T, d, d, L, dtype="bf16", seed=seed))
        with B.Plan.for_inputs(inp, path=2, segments=P) as plan:
            ref = plan.forward(inp, stream=stream)
        out = torch.full_like(inp["v"], float("nan"))
        status = B.prism_forward_noalloc(Bn, H, T, d, d, L, inp["q"], inp["k"], inp["v"], inp["beta"],
                                         inp["alpha"], inp["u"], inp["gamma"], inp["eta"], inp["conv_w"], out,
                                         stream=stream)
        torch.cuda.synchronize()
        assert status == 0
        assert torch.isfinite(out.float()).all()
        err = rel_err(out.double().cpu().numpy(), ref.double().cpu().numpy())
        assert err <= TOL["bf16"], err


def test_noalloc_rejects_sizes_beyond_its_scratch():
    build.build()
    lib = B.lib()
    # 64 MiB cannot hold the per-chunk stash of 64 sequences x 64K tokens
    rc = lib.prism_forward_noalloc(8, 8, 65536, 64, 64, 4, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, None, None)
    assert rc == B.PRISM_ERR_UNSUPPORTED
    assert "too large for the fixed scratch" in B.prism_last_error_message()
    rc = lib.prism_forward_noalloc(1, 1, 64, 128, 128, 2, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, None, None)
    assert rc == B.PRISM_ERR_UNSUPPORTED
