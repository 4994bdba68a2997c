"""CPU checks of the C ABI: the library loads, exports every function that
include/lopt.h declares, and argument validation that needs no device
returns the documented error codes.  No compute call is made."""

import ctypes
import os
import re

import numpy as np

import pytest

from learned_optimizer_step_gb300 import build as B
from learned_optimizer_step_gb300 import lopt as L

HEADER = os.path.join(B.ROOT, "include", "lopt.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lopt_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("lopt_create", "lopt_step", "lopt_destroy", "lopt_strerror"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), "liblopt.so does not export " + name
    assert sorted(declared_functions()) == sorted(L.EXPORTED)


def test_struct_layout_matches_header():
    # 12 pointers, two int64 and two int32, natural alignment, no padding
    assert ctypes.sizeof(L.LoptTensor) == 12 * 8 + 2 * 8 + 2 * 4
    assert L.LoptTensor.rows.offset == 96


def test_error_strings(lib):
    for code, name in L.ERRORS.items():
        s = lib.lopt_strerror(code).decode()
        assert s and s != "unknown error", name
    assert lib.lopt_strerror(0).decode() == "ok"
    assert lib.lopt_version() >= 100


def test_weight_set_size(lib):
    assert lib.lopt_weight_set_size(39, 32) == 39 * 32 + 32 + 32 * 32 + 32 + 64 + 2
    assert lib.lopt_weight_set_size(39, 4) == 39 * 4 + 4 + 16 + 4 + 8 + 2
    assert lib.lopt_weight_set_size(30, 32) == -1
    assert lib.lopt_weight_set_size(39, 0) == -1


def test_validation_before_any_device_call(lib):
    h = ctypes.c_void_p()
    w = (ctypes.c_float * 10)()
    fp = ctypes.cast(w, ctypes.POINTER(ctypes.c_float))
    assert lib.lopt_create(fp, 39, 32, 1, None) == -1
    assert lib.lopt_create(None, 39, 32, 1, ctypes.byref(h)) == -1
    assert lib.lopt_create(fp, 30, 32, 1, ctypes.byref(h)) == -1
    assert lib.lopt_create(fp, 39, 32, 0, ctypes.byref(h)) == -1
    assert lib.lopt_create(fp, 39, 65, 1, ctypes.byref(h)) == -6
    assert h.value is None
    assert lib.lopt_step(None, None, 0, 1, 1.0, None) == -1
    assert lib.lopt_step_host(None, None, 0, None, None, 1, 1.0, None) == -1
    assert lib.lopt_host_sync(None, None) == -1
    assert lib.lopt_set_host_groups(None, 4) == -1
    assert isinstance(lib.lopt_last_cuda_error(), bytes)
    assert lib.lopt_check(None) == -1
    assert lib.lopt_destroy(None) == -1
    assert lib.lopt_set_mlp_path(None, 0) == -1
    assert lib.lopt_set_weight_decay(None, 0.0) == -1
    assert lib.lopt_set_sweep_bytes(None, 0) == -1
    assert lib.lopt_selftest_wait(0) == -1
    assert lib.lopt_selftest_wait(2_000_000_000) == -1
    assert lib.lopt_feature_stats(None, 0, None) == -1
    assert lib.lopt_set_kernel_timing(None, 1) == -1
    assert lib.lopt_kernel_times(None, None, None) == -1
    assert lib.lopt_rowcol_static(None, None, None, 4, 4, None, None) == -1
    n_units = (ctypes.c_int32 * 3)()
    n_groups = ctypes.c_int32()
    assert lib.lopt_schedule_info(None, 1, 0, n_units, None, None, ctypes.byref(n_groups), None) == -1
    assert lib.lopt_schedule_info(None, 0, 0, None, None, None, ctypes.byref(n_groups), None) == -1
    assert lib.lopt_schedule_info(None, 0, -1, n_units, None, None, ctypes.byref(n_groups), None) == -1
    bad = (L.LoptTensor * 1)()
    bad[0].rows, bad[0].cols, bad[0].reserved = 4, 4, 1
    assert lib.lopt_schedule_info(bad, 1, 0, n_units, None, None, ctypes.byref(n_groups), None) == -1


def test_binding_rejects_non_cuda_tensors():
    torch = pytest.importorskip("torch")
    t = torch.zeros(4)
    with pytest.raises(TypeError):
        L._ptr(t, 4, "param")


def test_binding_host_buffers_must_be_cpu_float32():
    torch = pytest.importorskip("torch")
    assert L._host_ptr(torch.zeros(4), 4, "g") != 0
    assert L._host_ptr(np.zeros(4, np.float32), 4, "g") != 0
    with pytest.raises(TypeError):
        L._host_ptr(torch.zeros(4, dtype=torch.float64), 4, "g")
    with pytest.raises(TypeError):
        L._host_ptr(np.zeros(4), 4, "g")
    with pytest.raises(ValueError):
        L._host_ptr(torch.zeros(5), 4, "g")
