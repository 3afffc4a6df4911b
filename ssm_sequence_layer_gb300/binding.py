"""Thin ctypes binding of the C ABI in ``include/prism.h``.

Argument marshalling only: every step of the forward runs in the CUDA library
``libprism_gb300.so``.  The functions keep the C names.  Tensors are passed as
``torch.Tensor`` (device memory for ``prism_forward``, ``prism_forward_state`` and
``prism_decode_step``, host memory for ``prism_forward_host``) or as raw integer addresses.  There is no fallback: if
the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

PRISM_OK = 0
PRISM_ERR_INVALID_ARG = 1
PRISM_ERR_UNSUPPORTED = 2
PRISM_ERR_MISALIGNED = 3
PRISM_ERR_ARCH = 4
PRISM_ERR_CUDA = 5
PRISM_ERR_TIMEOUT = 6
PRISM_ERR_DEVICE = 7

PRISM_F32 = 0
PRISM_BF16 = 1

PRISM_OPT_SEGMENTS = 0
PRISM_OPT_PATH = 1
PRISM_OPT_WAIT_NS = 2
PRISM_OPT_TIMING = 3
PRISM_OPT_OUT_DTYPE = 4

EXPORTED = ("prism_plan", "prism_plan_set_option", "prism_forward", "prism_forward_host",
            "prism_plan_destroy", "prism_workspace_bytes", "prism_plan_last_device_status",
            "prism_status_string", "prism_last_error_message", "prism_version", "prism_plan_kernel_times",
            "prism_forward_noalloc", "prism_forward_state", "prism_decode_step", "prism_forward_nonlinear",
            "prism_project", "prism_backward", "prism_backward_nonlinear")


class prism_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("ms", ctypes.c_float)]

_lock = threading.Lock()
_LIB = None


class PrismError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{prism_status_string(status)} -- {message}")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _LIB
    with _lock:
        if _LIB is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{os.path.basename(path)} is not built; run "
                                   "`python -m ssm_sequence_layer_gb300.build` (needs nvcc)")
            L = ctypes.CDLL(path)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
            L.prism_plan.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(vp)]
            L.prism_plan_set_option.argtypes = [vp, i, ctypes.c_longlong]
            fwd = [vp, vp, vp, vp, f, f, vp, f, f, vp, i, vp, vp]
            L.prism_forward.argtypes = fwd
            L.prism_forward_host.argtypes = fwd
            L.prism_plan_destroy.argtypes = [vp]
            L.prism_workspace_bytes.argtypes = [vp]
            L.prism_workspace_bytes.restype = ctypes.c_size_t
            L.prism_plan_last_device_status.argtypes = [vp]
            L.prism_status_string.argtypes = [i]
            L.prism_status_string.restype = ctypes.c_char_p
            L.prism_last_error_message.restype = ctypes.c_char_p
            L.prism_version.restype = ctypes.c_char_p
            L.prism_plan_kernel_times.argtypes = [vp, ctypes.POINTER(prism_kernel_time), i]
            L.prism_forward_noalloc.argtypes = [i] * 6 + [vp, vp, vp, f, f, vp, f, f, vp, vp, vp,
                                                          ctypes.POINTER(ctypes.c_int)]
            L.prism_forward_noalloc.restype = ctypes.c_int
            L.prism_forward_state.argtypes = fwd[:11] + [vp, f, vp, f, vp, vp]
            L.prism_decode_step.argtypes = fwd[:11] + [vp, f, vp, vp]
            L.prism_forward_nonlinear.argtypes = fwd[:11] + [vp, f, vp, f, vp, vp]
            L.prism_project.argtypes = [vp, i, vp, vp, vp, vp, vp, f, vp]
            L.prism_backward.argtypes = fwd[:11] + [vp, f, f, f] + [f] * 11 + [vp]
            L.prism_backward_nonlinear.argtypes = L.prism_backward.argtypes
            L.prism_plan_kernel_times.restype = ctypes.c_int
            for name in ("prism_plan", "prism_plan_set_option", "prism_forward", "prism_forward_host",
                         "prism_plan_destroy", "prism_plan_last_device_status", "prism_forward_state",
                         "prism_decode_step", "prism_forward_nonlinear", "prism_project", "prism_backward",
                         "prism_backward_nonlinear"):
                getattr(L, name).restype = ctypes.c_int
            _LIB = L
    return _LIB


def _check(status):
    if status != PRISM_OK:
        raise PrismError(status, prism_last_error_message())
    return status


def _addr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def prism_status_string(status: int) -> str:
    return lib().prism_status_string(int(status)).decode()


def prism_last_error_message() -> str:
    return lib().prism_last_error_message().decode()


def prism_version() -> str:
    return lib().prism_version().decode()


def prism_plan(B, H, T, dk, dv, L, io=PRISM_BF16) -> int:
    h = ctypes.c_void_p()
    _check(lib().prism_plan(B, H, T, dk, dv, L, int(io), ctypes.byref(h)))
    return h.value


def prism_plan_set_option(plan, opt, value):
    return _check(lib().prism_plan_set_option(plan, int(opt), int(value)))


def prism_plan_destroy(plan):
    return _check(lib().prism_plan_destroy(plan))


def prism_workspace_bytes(plan) -> int:
    return int(lib().prism_workspace_bytes(plan))


def prism_plan_last_device_status(plan):
    return _check(lib().prism_plan_last_device_status(plan))


def prism_plan_kernel_times(plan, max_kernels=16):
    """[(name, ms), ...] of the last forward (ms = -1 when timing was off)."""
    buf = (prism_kernel_time * max_kernels)()
    n = lib().prism_plan_kernel_times(plan, buf, max_kernels)
    if n < 0:
        raise PrismError(PRISM_ERR_INVALID_ARG, prism_last_error_message())
    return [(buf[i].name.decode(), float(buf[i].ms)) for i in range(min(n, max_kernels))]


def prism_forward(plan, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, out, stream=None):
    return _check(lib().prism_forward(plan, _addr(q), _addr(k), _addr(v), _addr(beta), _addr(alpha), _addr(u),
                                      _addr(gamma), _addr(eta), _addr(conv_w), int(L), _addr(out),
                                      _stream(stream)))


def prism_forward_host(plan, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, out, stream=None):
    return _check(lib().prism_forward_host(plan, _addr(q), _addr(k), _addr(v), _addr(beta), _addr(alpha),
                                           _addr(u), _addr(gamma), _addr(eta), _addr(conv_w), int(L), _addr(out),
                                           _stream(stream)))


def prism_forward_state(plan, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, v_hist, S_init, out, S_final,
                        v_hist_out, stream=None):
    return _check(lib().prism_forward_state(plan, _addr(q), _addr(k), _addr(v), _addr(beta), _addr(alpha),
                                            _addr(u), _addr(gamma), _addr(eta), _addr(conv_w), int(L),
                                            _addr(v_hist), _addr(S_init), _addr(out), _addr(S_final),
                                            _addr(v_hist_out), _stream(stream)))


def prism_forward_nonlinear(plan, q, k, v, beta, alpha, u, gamma, p_gain, conv_w, L, v_hist, S_init, out, S_final,
                            v_hist_out, stream=None):
    return _check(lib().prism_forward_nonlinear(plan, _addr(q), _addr(k), _addr(v), _addr(beta), _addr(alpha),
                                                _addr(u), _addr(gamma), _addr(p_gain), _addr(conv_w), int(L),
                                                _addr(v_hist), _addr(S_init), _addr(out), _addr(S_final),
                                                _addr(v_hist_out), _stream(stream)))


def prism_project(plan, D, X, conv_x, W, u, p, gamma, stream=None):
    return _check(lib().prism_project(plan, int(D), _addr(X), _addr(conv_x), _addr(W), _addr(u), _addr(p),
                                      _addr(gamma), _stream(stream)))


def prism_decode_step(plan, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, v_hist, S, out, stream=None):
    return _check(lib().prism_decode_step(plan, _addr(q), _addr(k), _addr(v), _addr(beta), _addr(alpha),
                                          _addr(u), _addr(gamma), _addr(eta), _addr(conv_w), int(L),
                                          _addr(v_hist), _addr(S), _addr(out), _stream(stream)))


def prism_backward(plan, q, k, v, beta, alpha, u, gamma, eta, conv_w, L, v_hist, S_init, dout, dS_final, dq, dk, dv,
                   dbeta, dalpha, du, dgamma, deta, dconv_w, dv_hist, dS_init, stream=None):
    return _check(lib().prism_backward(plan, _addr(q), _addr(k), _addr(v), _addr(beta), _addr(alpha), _addr(u),
                                       _addr(gamma), _addr(eta), _addr(conv_w), int(L), _addr(v_hist),
                                       _addr(S_init), _addr(dout), _addr(dS_final), _addr(dq), _addr(dk), _addr(dv),
                                       _addr(dbeta), _addr(dalpha), _addr(du), _addr(dgamma), _addr(deta),
                                       _addr(dconv_w), _addr(dv_hist), _addr(dS_init), _stream(stream)))


def prism_backward_nonlinear(plan, q, k, v, beta, alpha, u, gamma, p_gain, conv_w, L, v_hist, S_init, dout, dS_final,
                             dq, dk, dv, dbeta, dalpha, du, dgamma, dp_gain, dconv_w, dv_hist, dS_init, stream=None):
    return _check(lib().prism_backward_nonlinear(plan, _addr(q), _addr(k), _addr(v), _addr(beta), _addr(alpha),
                                                 _addr(u), _addr(gamma), _addr(p_gain), _addr(conv_w), int(L),
                                                 _addr(v_hist), _addr(S_init), _addr(dout), _addr(dS_final),
                                                 _addr(dq), _addr(dk), _addr(dv), _addr(dbeta), _addr(dalpha),
                                                 _addr(du), _addr(dgamma), _addr(dp_gain), _addr(dconv_w),
                                                 _addr(dv_hist), _addr(dS_init), _stream(stream)))


def prism_forward_noalloc(B, H, T, dk, dv, L, q, k, v, beta, alpha, u, gamma, eta, conv_w, out, stream=None,
                          wait=True):
    """The allocation-free forward (see include/prism.h).  With wait=True the call waits for
    the stream and returns the device status word (0 = no condition recorded)."""
    status = ctypes.c_int(0)
    _check(lib().prism_forward_noalloc(B, H, T, dk, dv, L, _addr(q), _addr(k), _addr(v), _addr(beta),
                                       _addr(alpha), _addr(u), _addr(gamma), _addr(eta), _addr(conv_w), _addr(out),
                                       _stream(stream), ctypes.byref(status) if wait else None))
    return status.value


# ------------------------------------------------------------------------------------------------
class Plan:
    """Owns a ``prism_plan_t``; ``forward`` marshals a dict of tensors into ``prism_forward``."""

    def __init__(self, B, H, T, dk, dv, L, io="bf16", segments=None, path=None, out=None):
        self.shape = (B, H, T, dk, dv, L)
        self.io = io
        self.out = out or io
        self.handle = prism_plan(B, H, T, dk, dv, L, PRISM_BF16 if io == "bf16" else PRISM_F32)
        if self.out != io:
            prism_plan_set_option(self.handle, PRISM_OPT_OUT_DTYPE, PRISM_BF16 if self.out == "bf16" else PRISM_F32)
        if segments is not None:
            prism_plan_set_option(self.handle, PRISM_OPT_SEGMENTS, segments)
        if path is not None:
            prism_plan_set_option(self.handle, PRISM_OPT_PATH, path)

    @classmethod
    def for_inputs(cls, inp, **kw):
        B, H, T, dk = inp["q"].shape
        dv = inp["v"].shape[-1]
        io = "bf16" if str(inp["q"].dtype).endswith("bfloat16") else "f32"
        return cls(B, H, T, dk, dv, inp["L"], io=io, **kw)

    def set_option(self, opt, value):
        prism_plan_set_option(self.handle, opt, value)

    def workspace_bytes(self):
        return prism_workspace_bytes(self.handle)

    def _tensors(self, inp):
        L = inp["L"]
        lv = L > 1
        return (inp["q"], inp["k"], inp["v"], inp["beta"], inp["alpha"], inp["u"] if lv else None,
                inp["gamma"] if lv else None, inp["eta"] if lv else None, inp["conv_w"], L)

    def forward(self, inp, out=None, stream=None):
        """Device tensors in, device tensor out (allocated if not given)."""
        import torch
        ts = self._tensors(inp)
        for t in ts[:-1]:
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError("prism_forward takes contiguous CUDA tensors")
        if out is None:
            out = torch.empty(inp["v"].shape, dtype=self._out_torch_dtype(), device=inp["v"].device)
        prism_forward(self.handle, *ts, out, stream)
        return out

    @staticmethod
    def _check_device(ts, what):
        for t in ts:
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise ValueError(f"{what} takes contiguous CUDA tensors")

    def forward_state(self, inp, v_hist=None, S_init=None, S_final=None, v_hist_out=None, out=None, stream=None):
        """One part of a sequence evaluated over consecutive calls (see prism_forward_state):
        v_hist [B,H,3,dv] and S_init [B,H,dv,dk] (fp32) carry the sequence in, S_final and
        v_hist_out carry it out (each may be None; S_final may be S_init, v_hist_out v_hist)."""
        import torch
        ts = self._tensors(inp)
        self._check_device(ts[:-1] + (v_hist, S_init, S_final, v_hist_out), "prism_forward_state")
        if out is None:
            out = torch.empty(inp["v"].shape, dtype=self._out_torch_dtype(), device=inp["v"].device)
        prism_forward_state(self.handle, *ts, v_hist, S_init, out, S_final, v_hist_out, stream)
        return out

    def forward_nonlinear(self, inp, p_gain, v_hist=None, S_init=None, S_final=None, v_hist_out=None, out=None,
                          stream=None):
        """The non-linear residual variant (see prism_forward_nonlinear): p_gain [B,H,T,R,dv] in
        the io dtype takes the place of eta; the state arguments are those of forward_state."""
        import torch
        q, k, v, beta, alpha, u, gamma, _eta, conv_w, L = self._tensors(inp)
        lv = L > 1
        self._check_device((q, k, v, beta, alpha, u, gamma, conv_w, p_gain if lv else None, v_hist, S_init,
                            S_final, v_hist_out), "prism_forward_nonlinear")
        if out is None:
            out = torch.empty(inp["v"].shape, dtype=self._out_torch_dtype(), device=inp["v"].device)
        prism_forward_nonlinear(self.handle, q, k, v, beta, alpha, u, gamma, p_gain if lv else None, conv_w, L,
                                v_hist, S_init, out, S_final, v_hist_out, stream)
        return out

    def project(self, X, conv_x, W, out=None, stream=None):
        """The block's input projections (see prism_project): X [B,T,D], conv_x [4,D], W [N,D],
        bf16 CUDA tensors; returns (u, p, gamma), allocated unless `out` gives them."""
        import torch
        self._check_device((X, conv_x, W), "prism_project")
        B, H, T, dk, dv, L = self.shape
        R = L - 1
        if out is None:
            dev = X.device
            out = (torch.empty(B, H, T, R, dk, dtype=torch.bfloat16, device=dev),
                   torch.empty(B, H, T, R, dv, dtype=torch.bfloat16, device=dev),
                   torch.empty(B, H, T, R, dtype=torch.float32, device=dev))
        u, p, gamma = out
        prism_project(self.handle, X.shape[-1], X, conv_x, W, u, p, gamma, stream)
        return u, p, gamma

    def decode_step(self, inp, v_hist, S, out=None, stream=None):
        """One token per sequence (see prism_decode_step): q, k [B,H,dk], v [B,H,dv], u [B,H,R,dk],
        beta, alpha [B,H], gamma, eta [B,H,R] (a T axis of length 1 is accepted too); v_hist and
        S are updated in place."""
        import torch
        ts = self._tensors(inp)
        self._check_device(ts[:-1] + (v_hist, S), "prism_decode_step")
        if out is None:
            B, H = self.shape[:2]
            out = torch.empty((B, H, self.shape[4]), dtype=self._out_torch_dtype(), device=inp["v"].device)
        prism_decode_step(self.handle, *ts, v_hist, S, out, stream)
        return out

    def backward(self, inp, dout, dS_final=None, v_hist=None, S_init=None, want_dv_hist=False,
                 want_dS_init=False, grads=None, stream=None, p_gain=None):
        """Cotangents of the inputs (see prism_backward): dout [B,H,T,dv] and dS_final
        [B,H,dv,dk] are float32 CUDA tensors (dS_final may be None).  Returns a dict of float32
        tensors dq, dk, dv, dbeta, dalpha, du, dgamma, deta, dconv_w (plus dv_hist and dS_init on
        request), allocated unless `grads` holds them.  With p_gain [B,H,T,R,dv] (io dtype) the
        forward is the non-linear residual variant (see prism_backward_nonlinear): eta is not read
        and dp_gain [B,H,T,R,dv] takes the place of deta."""
        import torch
        ts = self._tensors(inp)
        B, H, T, dk, dv, L = self.shape
        R = L - 1
        nl = p_gain is not None
        if nl:
            ts = ts[:7] + (None,) + ts[8:]
        self._check_device(ts[:-1] + (dout, dS_final, v_hist, S_init, p_gain if R > 0 else None), "prism_backward")
        if grads is None:
            dev = inp["v"].device
            e = lambda *shape: torch.empty(*shape, dtype=torch.float32, device=dev)  # noqa: E731
            grads = {"dq": e(B, H, T, dk), "dk": e(B, H, T, dk), "dv": e(B, H, T, dv), "dbeta": e(B, H, T),
                     "dalpha": e(B, H, T), "du": e(B, H, T, R, dk), "dgamma": e(B, H, T, R),
                     ("dp_gain" if nl else "deta"): e(B, H, T, R, dv) if nl else e(B, H, T, R),
                     "dconv_w": e(H, 4, dv)}
            if want_dv_hist:
                grads["dv_hist"] = e(B, H, 3, dv)
            if want_dS_init:
                grads["dS_init"] = e(B, H, dv, dk)
        g = grads
        lv = R > 0
        self._check_device(tuple(g.values()), "prism_backward")
        if nl:
            q, k, v, beta, alpha, u, gamma, _eta, conv_w, L = ts
            prism_backward_nonlinear(self.handle, q, k, v, beta, alpha, u, gamma, p_gain if lv else None, conv_w, L,
                                     v_hist, S_init, dout, dS_final, g["dq"], g["dk"], g["dv"], g["dbeta"],
                                     g["dalpha"], g["du"] if lv else None, g["dgamma"] if lv else None,
                                     g["dp_gain"] if lv else None, g["dconv_w"], g.get("dv_hist"), g.get("dS_init"),
                                     stream)
            return g
        prism_backward(self.handle, *ts, v_hist, S_init, dout, dS_final, g["dq"], g["dk"], g["dv"], g["dbeta"],
                       g["dalpha"], g["du"] if lv else None, g["dgamma"] if lv else None, g["deta"] if lv else None,
                       g["dconv_w"], g.get("dv_hist"), g.get("dS_init"), stream)
        return g

    def _out_torch_dtype(self):
        import torch
        return torch.bfloat16 if self.out == "bf16" else torch.float32

    def forward_host(self, inp, out=None, stream=None):
        """Host tensors in (pinned for speed), host tensor out; synchronous."""
        import torch
        ts = self._tensors(inp)
        for t in ts[:-1]:
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("prism_forward_host takes contiguous host tensors")
        if out is None:
            out = torch.empty(inp["v"].shape, dtype=self._out_torch_dtype())
        prism_forward_host(self.handle, *ts, out, stream)
        return out

    def kernel_times(self):
        return prism_plan_kernel_times(self.handle)

    def last_device_status(self):
        return prism_plan_last_device_status(self.handle)

    def close(self):
        if self.handle:
            prism_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()
