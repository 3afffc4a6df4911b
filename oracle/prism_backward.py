"""Python front end of the fp64 CPU oracle for the PRISM recurrence's backward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library (``ssm_sequence_layer_gb300``) and never imports it.

The arithmetic lives in ``prism_oracle_bwd.c`` (reverse-mode differentiation of the
sequential fp64 definition, token by token; the header of that file states every
step).  This module compiles that file with gcc and calls it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from .prism_oracle import _f64, _ptr, build

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "prism_oracle_bwd.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libprism_oracle_bwd.so")
_lock = threading.Lock()
_lib = None

GRAD_NAMES = ("q", "k", "v", "beta", "alpha", "u", "gamma", "eta", "conv_w")


def build_backward(force: bool = False) -> str:
    return build(force=force, src=_SRC, lib_path=_LIB_PATH)


def _open(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.prism_oracle_backward_f64.restype = ctypes.c_int
    lib.prism_oracle_backward_f64.argtypes = [ctypes.c_int] * 6 + [dp] * 14 + [dp] * 12 + [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build_backward())
    return _lib


class BackwardLib:
    """The same front end bound to another build of the backward source (the tests that plant
    mistakes in a copy of it use this)."""

    def __init__(self, lib_path):
        self._lib = _open(lib_path)

    def backward(self, *args, **kw):
        return _backward(self._lib, *args, **kw)


def backward(q, k, v, beta, alpha, u, gamma, eta, conv_w, L, dout, *, S_init=None, v_hist=None, dS_final=None,
             p_gain=None, want_dv_hist=False, want_dS_init=False, nthreads=None):
    """Cotangents of every input of the linear-chain forward, given ``dout`` = dLoss/d out
    [B,H,T,dv] and optionally ``dS_final`` = dLoss/d S_final [B,H,dv,dk].

    Returns a dict with ``dq``, ``dk``, ``dv``, ``dbeta``, ``dalpha``, ``du``, ``dgamma``,
    ``deta``, ``dconv_w`` (each with its input's layout; the level tensors are [..,0] shaped
    when L = 1) and, on request, ``dv_hist`` [B,H,3,dv] and ``dS_init`` [B,H,dv,dk], all fp64.
    With ``p_gain`` [B,H,T,R,dv] the forward is the non-linear residual variant (``eta`` is not
    read and may be None) and ``dp_gain`` takes the place of ``deta``.
    """
    return _backward(_load(), q, k, v, beta, alpha, u, gamma, eta, conv_w, L, dout, S_init=S_init, v_hist=v_hist,
                     dS_final=dS_final, p_gain=p_gain, want_dv_hist=want_dv_hist, want_dS_init=want_dS_init,
                     nthreads=nthreads)


def _backward(lib, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, dout, *, S_init=None, v_hist=None,
              dS_final=None, p_gain=None, want_dv_hist=False, want_dS_init=False, nthreads=None):
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    beta, alpha, conv_w = _f64(beta), _f64(alpha), _f64(conv_w)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    R = L - 1
    if R > 0:
        u, gamma, eta, p_gain = _f64(u), _f64(gamma), _f64(eta), _f64(p_gain)
        assert u.shape == (B, H, T, R, dk) and gamma.shape == (B, H, T, R)
        assert (eta is None and p_gain is not None) or eta.shape == (B, H, T, R)
        assert p_gain is None or p_gain.shape == (B, H, T, R, dv)
        if p_gain is not None:
            eta = None
    else:
        u = gamma = eta = p_gain = None
    assert k.shape == (B, H, T, dk) and v.shape == (B, H, T, dv) and dout.shape == (B, H, T, dv)
    assert beta.shape == (B, H, T) and alpha.shape == (B, H, T) and conv_w.shape == (H, 4, dv)
    S_init, v_hist, dS_final = _f64(S_init), _f64(v_hist), _f64(dS_final)
    for name, x, shp in (("S_init", S_init, (B, H, dv, dk)), ("v_hist", v_hist, (B, H, 3, dv)),
                         ("dS_final", dS_final, (B, H, dv, dk))):
        assert x is None or x.shape == shp, f"{name} has shape {x.shape}, expected {shp}"
    g = {
        "dq": np.zeros((B, H, T, dk)), "dk": np.zeros((B, H, T, dk)), "dv": np.zeros((B, H, T, dv)),
        "dbeta": np.zeros((B, H, T)), "dalpha": np.zeros((B, H, T)),
        "du": np.zeros((B, H, T, R, dk)), "dgamma": np.zeros((B, H, T, R)), "deta": np.zeros((B, H, T, R)),
        "dconv_w": np.zeros((H, 4, dv)),
    }
    nonlinear = p_gain is not None
    if nonlinear:
        del g["deta"]
        g["dp_gain"] = np.zeros((B, H, T, R, dv))
    dvh = np.zeros((B, H, 3, dv)) if want_dv_hist else None
    dSi = np.zeros((B, H, dv, dk)) if want_dS_init else None
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    lvl = R > 0
    rc = lib.prism_oracle_backward_f64(
        B, H, T, dk, dv, L, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(u), _ptr(gamma), _ptr(eta),
        _ptr(p_gain), _ptr(conv_w), _ptr(v_hist), _ptr(S_init), _ptr(dout), _ptr(dS_final),
        _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dbeta"]), _ptr(g["dalpha"]),
        _ptr(g["du"]) if lvl else None, _ptr(g["dgamma"]) if lvl else None,
        _ptr(g["deta"]) if lvl and not nonlinear else None, _ptr(g.get("dp_gain")) if lvl else None,
        _ptr(g["dconv_w"]), _ptr(dvh), _ptr(dSi), int(nthreads))
    if rc != 0:
        raise ValueError(f"backward oracle failed (code {rc})")
    if want_dv_hist:
        g["dv_hist"] = dvh
    if want_dS_init:
        g["dS_init"] = dSi
    return g
