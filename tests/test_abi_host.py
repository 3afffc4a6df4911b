"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/prism.h declares, its enums match the binding, and argument
validation rejects bad sizes before touching a device."""
import ctypes
import os
import re

import pytest
import torch

from ssm_sequence_layer_gb300 import binding as B
from ssm_sequence_layer_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "prism.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.lib()


def header_functions():
    text = open(HEADER).read()
    return re.findall(r"PRISM_API\s+[\w\s\*]+?\b(prism_\w+)\s*\(", text)


def header_enum(name):
    text = open(HEADER).read()
    body = re.search(r"typedef enum %s \{(.*?)\}" % name, text, re.S).group(1)
    return {k: int(v) for k, v in re.findall(r"(PRISM_\w+)\s*=\s*(\d+)", body)}


def test_every_declared_function_is_exported(lib):
    names = header_functions()
    assert len(names) == len(set(names)) >= 10
    for n in names:
        assert hasattr(lib, n), f"{n} declared in prism.h but not exported"
    assert set(names) == set(B.EXPORTED)


def test_no_undeclared_prism_exports(lib):
    out = os.popen(f"nm -D --defined-only {B.library_path()}").read()
    exported = set(re.findall(r"\b(prism_\w+)\b", out))
    assert exported == set(header_functions())


def test_enums_match_binding():
    for k, v in {**header_enum("prism_status"), **header_enum("prism_dtype"), **header_enum("prism_option")}.items():
        assert getattr(B, k) == v, k


def test_status_strings(lib):
    for k, v in header_enum("prism_status").items():
        assert B.prism_status_string(v).startswith(k)
    assert "unknown" in B.prism_status_string(99)
    assert re.fullmatch(r"\d+\.\d+\.\d+", B.prism_version())


@pytest.mark.parametrize("args,status", [
    ((0, 1, 16, 64, 64, 1), B.PRISM_ERR_INVALID_ARG),
    ((1, 0, 16, 64, 64, 1), B.PRISM_ERR_INVALID_ARG),
    ((1, 1, 0, 64, 64, 1), B.PRISM_ERR_INVALID_ARG),
    ((1, 1, 16, 64, 64, 0), B.PRISM_ERR_INVALID_ARG),
    ((1, 1, 16, 96, 64, 1), B.PRISM_ERR_UNSUPPORTED),
    ((1, 1, 16, 64, 32, 1), B.PRISM_ERR_UNSUPPORTED),
    ((1, 1, 16, 64, 64, 17), B.PRISM_ERR_UNSUPPORTED),
    ((300, 300, 16, 64, 64, 1), B.PRISM_ERR_UNSUPPORTED),
])
def test_plan_rejects_bad_sizes_before_touching_a_device(lib, args, status):
    h = ctypes.c_void_p(1234)
    rc = lib.prism_plan(*args, B.PRISM_BF16, ctypes.byref(h))
    assert rc == status
    assert h.value is None
    assert B.prism_last_error_message()


def test_plan_rejects_unknown_dtype(lib):
    h = ctypes.c_void_p()
    assert lib.prism_plan(1, 1, 16, 64, 64, 1, 7, ctypes.byref(h)) == B.PRISM_ERR_INVALID_ARG
    assert lib.prism_plan(1, 1, 16, 64, 64, 1, 0, None) == B.PRISM_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_plan_without_a_gpu_reports_cuda_error(lib):
    h = ctypes.c_void_p()
    rc = lib.prism_plan(1, 1, 16, 64, 64, 1, B.PRISM_BF16, ctypes.byref(h))
    assert rc in (B.PRISM_ERR_CUDA, B.PRISM_ERR_ARCH)
    assert h.value is None


def test_null_plan_handling(lib):
    assert lib.prism_plan_destroy(None) == B.PRISM_OK
    assert lib.prism_workspace_bytes(None) == 0
    assert lib.prism_plan_last_device_status(None) == B.PRISM_ERR_INVALID_ARG
    assert lib.prism_plan_set_option(None, 0, 1) == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_forward(None, 16, 16, 16, 16, 16, None, None, None, 16, 1, 16, None)
    assert rc == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_forward_host(None, 16, 16, 16, 16, 16, None, None, None, 16, 1, 16, None)
    assert rc == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_forward_state(None, 16, 16, 16, 16, 16, None, None, None, 16, 1, None, None, 16, None, None,
                                 None)
    assert rc == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_decode_step(None, 16, 16, 16, 16, 16, None, None, None, 16, 1, 16, 16, 16, None)
    assert rc == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_project(None, 64, 16, 16, 16, 16, 16, 16, None)
    assert rc == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_forward_nonlinear(None, 16, 16, 16, 16, 16, None, None, None, 16, 1, None, None, 16, None,
                                     None, None)
    assert rc == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_backward(None, 16, 16, 16, 16, 16, None, None, None, 16, 1, None, None, 16, None,
                            16, 16, 16, 16, 16, None, None, None, 16, None, None, None)
    assert rc == B.PRISM_ERR_INVALID_ARG
    rc = lib.prism_backward_nonlinear(None, 16, 16, 16, 16, 16, None, None, None, 16, 1, None, None, 16, None,
                                      16, 16, 16, 16, 16, None, None, None, 16, None, None, None)
    assert rc == B.PRISM_ERR_INVALID_ARG


def test_binding_raises_with_message(lib):
    with pytest.raises(B.PrismError) as ei:
        B.prism_plan(1, 1, 16, 80, 64, 1)
    assert ei.value.status == B.PRISM_ERR_UNSUPPORTED
    assert "dk and dv must be 64 or 128" in str(ei.value)
