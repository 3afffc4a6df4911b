"""Python front end of the fp64 CPU oracle for the PRISM memory-recurrence forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA library (``ssm_sequence_layer_gb300``) and never imports it.

The arithmetic lives in ``prism_oracle.c`` (a plain sequential loop over tokens in
fp64; the header of that file states the definition and where each step comes
from).  This module only compiles that file with gcc, marshals numpy arrays to
float64 and calls it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "prism_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libprism_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, lib_path: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (no fast-math, so erf/exp follow libm)."""
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    stale = (not os.path.exists(lib_path)) or os.path.getmtime(lib_path) < os.path.getmtime(src)
    if force or stale:
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
               src, "-o", tmp, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


def _open(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.prism_oracle_forward_f64.restype = ctypes.c_int
    lib.prism_oracle_forward_f64.argtypes = [ctypes.c_int] * 6 + [dp] * 12 + [dp] * 6 + [ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build())
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> numpy without importing torch here
        x = x.detach().float().cpu().numpy() if x.dtype.is_floating_point else x.cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def forward(q, k, v, beta, alpha, u, gamma, eta, conv_w, L, *, S_init=None, v_hist=None, p_gain=None,
            want_state=False, want_x=False, want_hge=False, nthreads=None):
    """Run the oracle.  Arrays follow the layouts in ``prism_oracle.c``; ``S_init``
    [B,H,dv,dk] and ``v_hist`` [B,H,3,dv] (v_{-3}, v_{-2}, v_{-1}) carry a sequence over
    from a previous call.  ``p_gain`` [B,H,T,R,dv] selects the non-linear residual variant
    (``eta`` is then not read and may be None).

    Returns a dict with ``out`` [B,H,T,dv] and, on request, ``S_final``
    [B,H,dv,dk], ``X`` [B,H,T,R,dv] and ``h``/``g``/``e`` [B,H,T,dv], all fp64.
    """
    return _forward(_load(), q, k, v, beta, alpha, u, gamma, eta, conv_w, L, S_init=S_init, v_hist=v_hist,
                    p_gain=p_gain, want_state=want_state, want_x=want_x, want_hge=want_hge, nthreads=nthreads)


class OracleLib:
    """The same front end bound to another build of the oracle source (used by the
    tests that plant mistakes in a copy of the source to show the pins catch them)."""

    def __init__(self, lib_path):
        self._lib = _open(lib_path)

    def forward(self, *args, **kw):
        return _forward(self._lib, *args, **kw)


def _forward(lib, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, *, S_init=None, v_hist=None, p_gain=None,
             want_state=False, want_x=False, want_hge=False, nthreads=None):
    q, k, v = _f64(q), _f64(k), _f64(v)
    beta, alpha, conv_w = _f64(beta), _f64(alpha), _f64(conv_w)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    R = L - 1
    if R > 0:
        u, gamma, eta, p_gain = _f64(u), _f64(gamma), _f64(eta), _f64(p_gain)
        assert u.shape == (B, H, T, R, dk) and gamma.shape == (B, H, T, R)
        assert (eta is None and p_gain is not None) or eta.shape == (B, H, T, R)
        assert p_gain is None or p_gain.shape == (B, H, T, R, dv)
    else:
        u = gamma = eta = p_gain = None
    assert k.shape == (B, H, T, dk) and v.shape == (B, H, T, dv)
    assert beta.shape == (B, H, T) and alpha.shape == (B, H, T) and conv_w.shape == (H, 4, dv)
    S_init = _f64(S_init)
    if S_init is not None:
        assert S_init.shape == (B, H, dv, dk)
    v_hist = _f64(v_hist)
    if v_hist is not None:
        assert v_hist.shape == (B, H, 3, dv)
    out = np.zeros((B, H, T, dv))
    S_final = np.zeros((B, H, dv, dk)) if want_state else None
    X = np.zeros((B, H, T, max(R, 0), dv)) if (want_x and R > 0) else None
    hh = np.zeros((B, H, T, dv)) if want_hge else None
    gg = np.zeros((B, H, T, dv)) if want_hge else None
    ee = np.zeros((B, H, T, dv)) if want_hge else None
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.prism_oracle_forward_f64(
        B, H, T, dk, dv, L, _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha), _ptr(u),
        _ptr(gamma), _ptr(eta), _ptr(p_gain), _ptr(conv_w), _ptr(v_hist), _ptr(S_init), _ptr(out), _ptr(S_final), _ptr(X),
        _ptr(hh), _ptr(gg), _ptr(ee), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    res = {"out": out}
    if want_state:
        res["S_final"] = S_final
    if want_x:
        res["X"] = X if X is not None else np.zeros((B, H, T, 0, dv))
    if want_hge:
        res.update(h=hh, g=gg, e=ee)
    return res
