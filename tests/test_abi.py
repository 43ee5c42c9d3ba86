"""The C-ABI library loads on a host without a GPU and exports every
function include/ffa.h declares; the binding refuses to run without CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from flexible_mask_attention_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ffa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(ffa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("ffa_plan_create", "ffa_plan_destroy", "ffa_fwd", "ffa_bwd",
              "ffa_fwd_workspace_size", "ffa_bwd_workspace_size", "ffa_plan_export",
              "ffa_get_last_device_error"):
        assert n in names


def test_every_declared_function_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in ffa.h but not exported"


def test_binding_names_match_header():
    import flexible_mask_attention_gb300 as ffa
    assert sorted(ffa.EXPORTED_SYMBOLS) == declared_functions()


def test_status_strings(lib):
    lib.ffa_status_string.restype = ctypes.c_char_p
    lib.ffa_status_string.argtypes = [ctypes.c_int32]
    assert lib.ffa_status_string(0) == b"ok"
    assert b"overlap" in lib.ffa_status_string(3)


def test_null_arguments_rejected_without_gpu(lib):
    """Argument checks run before any CUDA call."""
    P = ctypes.c_void_p
    lib.ffa_plan_create.argtypes = [ctypes.POINTER(P), P, P, P] + [ctypes.c_int32] * 8 + [P]
    assert lib.ffa_plan_create(None, None, None, None, 0, 1, 1, 1, 1, 128, 0, 0, None) == 1
    h = P()
    # unsupported head_dim is refused before the device is touched
    assert lib.ffa_plan_create(ctypes.byref(h), None, None, None, 0, 16, 16, 1, 1, 96, 0, 0,
                               None) == 4
    lib.ffa_fwd.argtypes = [P] * 4 + [ctypes.c_float] + [P] * 3 + [ctypes.c_size_t, P]
    assert lib.ffa_fwd(None, None, None, None, 0.0, None, None, None, 0, None) == 1


def test_product_path_fails_loudly_without_cuda():
    import torch
    import flexible_mask_attention_gb300 as ffa
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(Exception):
        ffa.ffa_plan_create([[0, 8]], [[0, 8]], [0], 8, 8, 1, 1, 128)
