"""Helpers shared by the GPU parity tests (not a test module)."""
import numpy as np
import torch

from ssm_sequence_layer_gb300 import binding as B

# max|o - o_ref| / rms(o_ref) over the compared outputs.  The bar measures the computation, so
# outputs are compared in fp32 (PRISM_OPT_OUT_DTYPE = float32): rounding a bf16 output alone
# costs up to 2^-9 max|o| / rms(o), which is 3.3e-2 on the 130M-LM layer shape.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_device(inp, device="cuda"):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in inp.items()}


def io_of(inp):
    return "bf16" if inp["q"].dtype == torch.bfloat16 else "f32"


def rel_err(out, ref):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(out - ref)) / max(rms, 1e-300))


def gpu_forward(inp, out="f32", **plan_kw):
    """Run prism_forward through the C ABI (fp32 output by default); returns fp64 numpy."""
    d = to_device(inp)
    with B.Plan.for_inputs(d, out=out, **plan_kw) as p:
        out = p.forward(d)
        torch.cuda.synchronize()
        p.last_device_status()
    return out.double().cpu().numpy()


def oracle_forward(oracle_mod, inp, **kw):
    return oracle_mod.forward(inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"],
                              inp["gamma"], inp["eta"], inp["conv_w"], inp["L"], **kw)


def bf16_half_ulp(x):
    """Half the spacing of bf16 numbers at |x| (8 significant bits): the largest error that
    rounding a value of that magnitude to bf16 can introduce."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-300)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def rel_err_bf16_out(out, ref):
    """max over elements of (|o - o_ref| minus the bf16 rounding allowance of that element) /
    rms(o_ref), for an output written in bf16.  Each element may differ from the fp64 reference by
    the half-ulp its own rounding to bf16 costs (taken at the larger of |o| and |o_ref|, so an
    element on a binade boundary keeps the wider spacing); what exceeds that is the computation's
    error, held to the same 2e-2 bar as the fp32 outputs."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    excess = np.maximum(np.abs(out - ref) - bf16_half_ulp(np.maximum(np.abs(out), np.abs(ref))), 0.0)
    return float(np.max(excess) / max(rms, 1e-300))
