"""Input projections of the PRISM block -- fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this module.  It shares no code with the CUDA library.

What it computes (the reading notes on PRISM, section 2.3, "Input-Anchored Simulation": a
short causal convolution over the layer input gives the anchor, and per refinement level three
projections of the anchor give the basis k^(l), the gain p^(l) and the gate beta^(l)); per batch
b and token t, with the layer input X [B,T,D]:

    a_t            = sum_{j=0..3} w_j (.) X_{t-j}         depthwise, zero before t = 0
    u_{t,l}  (h)   = y / ||y||,  y = Wu[h,l] a_t  (dk)   the basis, unit length (0 if y = 0)
    p_{t,l}  (h)   = Wp[h,l] a_t                  (dv)   the gain
    gamma_{t,l}(h) = sigmoid(wg[h,l] . a_t)              the gate

These are the directions u, gains p and step gates gamma that the recurrence (prism_oracle)
takes as inputs.  Weight layout W [N, D], N = H R dk + H R dv + H R: the rows of Wu in (h, l, c)
order, then those of Wp, then the H R gate rows.  conv_x [4, D] (tap j multiplies X_{t-j}).
Outputs: u [B,H,T,R,dk], p [B,H,T,R,dv], gamma [B,H,T,R], all fp64.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def anchor(X, conv_x):
    """a_t = sum_j w_j X_{t-j}, per batch, zero before the first token."""
    X, w = _f64(X), _f64(conv_x)
    B, T, D = X.shape
    a = np.zeros_like(X)
    for j in range(4):
        a[:, j:, :] += w[j][None, None, :] * X[:, : T - j, :]
    return a


def project(X, conv_x, W, H, R, dk, dv):
    """Returns (u, p, gamma) as described in the module docstring."""
    W = _f64(W)
    a = anchor(X, conv_x)
    B, T, D = a.shape
    NU, NP, NG = H * R * dk, H * R * dv, H * R
    assert W.shape == (NU + NP + NG, D)
    Y = a @ W.T  # [B, T, N]
    yu = Y[..., :NU].reshape(B, T, H, R, dk).transpose(0, 2, 1, 3, 4)
    norm = np.sqrt(np.sum(yu * yu, axis=-1, keepdims=True))
    u = np.where(norm > 0, yu / np.where(norm > 0, norm, 1.0), 0.0)
    p = Y[..., NU:NU + NP].reshape(B, T, H, R, dv).transpose(0, 2, 1, 3, 4)
    g = Y[..., NU + NP:].reshape(B, T, H, R).transpose(0, 2, 1, 3)
    gamma = 1.0 / (1.0 + np.exp(-g))
    return np.ascontiguousarray(u), np.ascontiguousarray(p), np.ascontiguousarray(gamma)
