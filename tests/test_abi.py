"""The C ABI library: builds, loads and exports every symbol its header
declares.  No compute call is made (these run without a GPU)."""
import ctypes
import pathlib
import os
import re

import pytest

import quantized_moe_expert_sigmoid_gb300 as moe
from quantized_moe_expert_sigmoid_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load_library()


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for n in ("moe_layer_create", "moe_route", "moe_forward", "moe_layer_forward_routed",
              "moe_layer_destroy", "moe_layer_check"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_python_binding_names_match_the_abi():
    for name in _declared_functions():
        assert callable(getattr(moe, name)), name


def test_status_strings(lib):
    for code, name in moe.STATUS.items():
        assert moe.moe_status_string(code) == name
    assert moe.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def _create(lib, **over):
    sh = dict(hidden=256, n_experts=8, top_k=2, expert_ffn=128, n_shared=1,
              routed_scaling=2.0, max_tokens=4, flags=0)
    sh.update(over)
    shapes = moe._Shapes(*(sh[k] for k, _ in moe._Shapes._fields_))
    w = moe._Weights(None, None, None, None, None, None)
    out = ctypes.c_void_p(12345)
    st = lib.moe_layer_create(ctypes.byref(shapes), ctypes.byref(w), None, ctypes.byref(out))
    return st, out.value


@pytest.mark.parametrize("over,status", [
    (dict(hidden=250), 2), (dict(hidden=0), 2), (dict(expert_ffn=48 + 1), 2),
    (dict(n_experts=0), 2), (dict(n_experts=300), 2), (dict(top_k=9), 2),
    (dict(top_k=9, n_experts=8), 2), (dict(n_shared=2), 2), (dict(max_tokens=0), 2),
    (dict(routed_scaling=0.0), 1), (dict(flags=16), 1), (dict(flags=0x80000001), 1), ({}, 1)])
def test_create_validates_before_touching_the_gpu(lib, over, status):
    st, handle = _create(lib, **over)
    assert st == status, moe.moe_last_error()
    assert handle is None
    assert moe.moe_last_error()
    if "flags" in over:
        assert "flags" in moe.moe_last_error()


@pytest.mark.parametrize("flags", [1, 2, 3, 4, 7, 8, 15])
def test_known_flags_are_accepted(lib, flags):
    # known flags pass the flags check and fail later, on the NULL weights
    st, handle = _create(lib, flags=flags)
    assert st == 1 and handle is None
    assert "flags" not in moe.moe_last_error()


def test_null_layer_rejected(lib):
    assert lib.moe_layer_check(None) == 1
    assert lib.moe_test_barrier_slack(None, 0) == 1
    assert lib.moe_layer_forward_routed_host(None, None, 0, 1, None, None, 0, None, None, None, 0, None) == 1
    assert lib.moe_route(None, None, 0, 0, None, None, 0, None, None, None) == 1
    assert lib.moe_forward(None, None, 0, 0, None, None, None, 0, None) == 1
    assert lib.moe_layer_forward_routed_resid(None, None, None, 1, None, None, 1e-6, 1, None, None, 0,
                                              None, None, None, 0, None) == 1
    assert lib.moe_layer_destroy(None) == 0
    assert lib.moe_layer_weight_bytes(None) == -1


def test_rmsnorm_argument_checks(lib):
    assert lib.moe_residual_rmsnorm(None, None, 1, None, 1, 12, 1e-6, None) == 1   # H % 8
    assert lib.moe_residual_rmsnorm(None, None, 1, None, -1, 16, 1e-6, None) == 1  # T < 0
    assert lib.moe_residual_rmsnorm(None, None, 1, None, 0, 16, 1e-6, None) == 0   # empty
    assert lib.moe_residual_rmsnorm(None, None, 1, None, 1, 16, 1e-6, None) == 1   # NULL
    assert lib.moe_residual_rmsnorm(ctypes.c_void_p(8), None, 1, ctypes.c_void_p(16), 1, 16,
                                    1e-6, None) == 3                                # misaligned


def test_stage_timing_argument_checks(lib):
    assert lib.moe_layer_enable_timing(None, 4) == 1      # NULL layer
    n = ctypes.c_int32(-1)
    assert lib.moe_layer_stage_times(None, None, 0, ctypes.byref(n)) == 1
    assert moe.STAGES == ("route+plan+gather", "up/gate", "down", "combine")


def test_flag_constants_match_the_header():
    src = (pathlib.Path(__file__).resolve().parents[1] / "include" / "moe_gb300.h").read_text()
    for name in ("MOE_FLAG_SELECTION_BIAS", "MOE_FLAG_DETERMINISTIC", "MOE_FLAG_HOST_IO", "MOE_FLAG_COOPERATIVE"):
        m = re.search(r"#define\s+%s\s+(\d+)u" % name, src)
        assert m and int(m.group(1)) == getattr(moe, name), name
