"""Seeded synthetic inputs for the PRISM memory-recurrence forward.

This module is shared by the CUDA path's tests and benchmark and by the oracle's
tests.  It draws random numbers and casts them; it holds none of the method's
arithmetic.

Recipe (every draw from one ``torch.Generator('cpu')`` seeded with ``seed``, in
this fixed order): q, k, v, beta, alpha, u, gamma, eta, conv_w.
  * q, k, u: standard Gaussian rows, each divided by its L2 norm over the
    feature dimension (so ||k|| = 1, the regime in which the GDN transition
    alpha (I - beta k k^T) is stable, notes on PRISM section 2.2);
  * v ~ N(0, 1);
  * beta, gamma, eta = sigmoid(N(0, 1)), all in (0, 1);
  * alpha = exp(-softplus(N(0, 1)) / alpha_div), alpha_div = 16 (64 for the
    long-memory workload);
  * conv_w ~ N(0, 1/4) (standard deviation 0.5), per head and channel.
All draws are fp32.  q, k, v, u and conv_w are then cast to the io dtype; the
gates (beta, alpha, gamma, eta) stay fp32.  With L = 1 there are no u, gamma or
eta draws.

The five named workloads reproduce the shapes the method is measured on: a tiny
fp32 case, a GDN-degenerate (L = 1) case, the 130M-parameter language-model
layer shape (2K tokens, 6 heads of 128), the 16K-token sequential-recommendation
shape (4 heads of 64) and a 64K-token long-memory stress case.  The decode
workloads take one token per sequence with those head shapes over a serving batch.
No dataset item is used: the values are synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    L: int
    dtype: str  # "f32" or "bf16": dtype of q, k, v, u, conv_w and out
    alpha_div: float = 16.0

    @property
    def R(self) -> int:
        return self.L - 1

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T

    def as_dict(self):
        return asdict(self)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 2, 256, 64, 64, 3, "f32"),
    "gdn_degenerate": Workload("gdn_degenerate", 4, 8, 2048, 128, 128, 1, "bf16"),
    "lm130m_layer": Workload("lm130m_layer", 8, 6, 2048, 128, 128, 4, "bf16"),
    "seqrec_16k": Workload("seqrec_16k", 2, 4, 16384, 64, 64, 4, "bf16"),
    "long_64k": Workload("long_64k", 1, 16, 65536, 128, 128, 8, "bf16", 64.0),
}
HEADLINE = "seqrec_16k"

# One recurrent step (one token per sequence) over a serving batch: the head shapes of the
# language-model layer and of the recommendation shape, with as many sequences as make the
# fp32 state (B H dv dk 4 bytes) larger than the 129 MB L2, so that a step streams it from HBM.
DECODE_WORKLOADS = {
    "decode_lm130m": Workload("decode_lm130m", 512, 6, 1, 128, 128, 4, "bf16"),
    "decode_seqrec": Workload("decode_seqrec", 2048, 4, 1, 64, 64, 4, "bf16"),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _unit_rows_(x: torch.Tensor) -> torch.Tensor:
    x.div_(x.norm(dim=-1, keepdim=True).clamp_min_(1e-30))
    return x


def make_inputs(B, H, T, dk, dv, L, dtype="bf16", seed=0, alpha_div=16.0):
    """Draw one input set (CPU tensors).  See the module docstring for the recipe."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    R = L - 1
    io = TORCH_DTYPE[dtype]
    f32 = torch.float32
    q = _unit_rows_(torch.randn(B, H, T, dk, generator=g, dtype=f32))
    k = _unit_rows_(torch.randn(B, H, T, dk, generator=g, dtype=f32))
    v = torch.randn(B, H, T, dv, generator=g, dtype=f32)
    beta = torch.sigmoid(torch.randn(B, H, T, generator=g, dtype=f32))
    alpha = torch.exp(-torch.nn.functional.softplus(torch.randn(B, H, T, generator=g, dtype=f32)) / alpha_div)
    if R > 0:
        u = _unit_rows_(torch.randn(B, H, T, R, dk, generator=g, dtype=f32))
        gamma = torch.sigmoid(torch.randn(B, H, T, R, generator=g, dtype=f32))
        eta = torch.sigmoid(torch.randn(B, H, T, R, generator=g, dtype=f32))
    else:
        u = torch.zeros(B, H, T, 0, dk, dtype=f32)
        gamma = torch.zeros(B, H, T, 0, dtype=f32)
        eta = torch.zeros(B, H, T, 0, dtype=f32)
    conv_w = torch.randn(H, 4, dv, generator=g, dtype=f32) * 0.5
    return {
        "q": q.to(io), "k": k.to(io), "v": v.to(io), "beta": beta, "alpha": alpha,
        "u": u.to(io), "gamma": gamma, "eta": eta, "conv_w": conv_w.to(io), "L": L,
    }


def make_workload_inputs(w: Workload | str, seed=0, **overrides):
    if isinstance(w, str):
        w = WORKLOADS[w]
    kw = dict(B=w.B, H=w.H, T=w.T, dk=w.dk, dv=w.dv, L=w.L, dtype=w.dtype, seed=seed,
              alpha_div=w.alpha_div)
    kw.update(overrides)
    return make_inputs(**kw)


def make_gain(B, H, T, L, dv, dtype="bf16", seed=0):
    """Gains p [B,H,T,L-1,dv] of the non-linear residual variant: sigmoid(N(0, 1)), the range
    of the gain GELU'(h) they stand in for, drawn from a generator of their own (seed + 7919)
    so that the other inputs of a seed are unchanged; cast to the io dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 7919)
    p = torch.sigmoid(torch.randn(B, H, T, max(L - 1, 0), dv, generator=g, dtype=torch.float32))
    return p.to(TORCH_DTYPE[dtype])


# The block's input projections: the layer input X [B,T,D] with D = H dk (the model width of the
# head shapes above), feeding R = L - 1 levels.
PROJECTION_WORKLOADS = {
    "project_seqrec": dict(B=2, T=16384, D=256, H=4, R=3, dk=64, dv=64),
    "project_lm130m": dict(B=8, T=2048, D=768, H=6, R=3, dk=128, dv=128),
}


def make_projection_inputs(B, T, D, H, R, dk, dv, seed=0):
    """X ~ N(0, 1) [B,T,D], conv_x ~ N(0, 1/4) [4,D], W ~ N(0, 1/D) [N,D] with
    N = H R (dk + dv + 1), drawn in that order from one generator, cast to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    N = H * R * (dk + dv + 1)
    X = torch.randn(B, T, D, generator=g)
    conv_x = torch.randn(4, D, generator=g) * 0.5
    W = torch.randn(N, D, generator=g) / D ** 0.5
    return {"X": X.to(torch.bfloat16), "conv_x": conv_x.to(torch.bfloat16), "W": W.to(torch.bfloat16),
            "B": B, "T": T, "D": D, "H": H, "R": R, "dk": dk, "dv": dv}


def select_heads(inp: dict, pairs):
    """Slice an input set down to the listed (b, h) pairs as a [1, len(pairs)] batch.

    Used to run the oracle on a sample of independent sequences of a large workload.
    """
    bs = torch.tensor([p[0] for p in pairs])
    hs = torch.tensor([p[1] for p in pairs])
    out = {"L": inp["L"]}
    for name in ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta"):
        out[name] = inp[name][bs, hs].unsqueeze(0)
    out["conv_w"] = inp["conv_w"][hs]
    return out


def make_cotangents(B, H, T, dk, dv, seed=0, with_state=False):
    """Cotangents for the backward pass: dout ~ N(0, 1) [B,H,T,dv] (float32) and, with
    ``with_state``, dS_final ~ N(0, 1) [B,H,dv,dk] (float32), drawn in that order from a
    generator of their own (seed + 104729) so that the forward inputs of a seed are unchanged."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 104729)
    dout = torch.randn(B, H, T, dv, generator=g, dtype=torch.float32)
    dS_final = torch.randn(B, H, dv, dk, generator=g, dtype=torch.float32) if with_state else None
    return dout, dS_final
