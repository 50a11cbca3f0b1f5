"""Host-side checks of the C ABI that need no GPU: the library builds, loads and exports every entry point
include/moe_block.h declares; calls with bad arguments or without a device fail with the documented status."""
import ctypes
import os
import re

import pytest

from w4a16_top_mixture_gb300 import build, lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe_block.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return lib.load_library()


def test_header_declares_entry_points():
    syms = declared_symbols()
    assert "moe_block_create" in syms and "moe_block_forward" in syms and len(syms) >= 10


def test_library_exports_every_declared_symbol(L):
    for s in declared_symbols():
        assert hasattr(L, s), s
    assert sorted(lib.EXPORTS) == declared_symbols()


def test_strerror_names_every_status(L):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert L.moe_block_strerror(s).decode() != "unknown status"


def test_invalid_arguments_without_device(L):
    h = ctypes.c_void_p()
    assert L.moe_block_create(None, ctypes.byref(h)) == -1
    cfg = lib.Config(2048, 256, 8, 512, 512, 64, 16)
    assert L.moe_block_create(ctypes.byref(cfg), None) == -1
    bad = lib.Config(2048, 256, 8, 512, 512, 32, 16)     # group size other than 64
    assert L.moe_block_create(ctypes.byref(bad), ctypes.byref(h)) == -2
    bad = lib.Config(3000, 256, 8, 512, 512, 64, 16)     # hidden without a kernel
    assert L.moe_block_create(ctypes.byref(bad), ctypes.byref(h)) == -2
    bad = lib.Config(2048, 256, 300, 512, 512, 64, 16)   # k > E
    assert L.moe_block_create(ctypes.byref(bad), ctypes.byref(h)) == -2
    assert L.moe_block_forward(None, None, None, 1, None) == -1
    assert L.moe_block_get_status(None, None) == -1


def test_create_without_gpu_reports_no_device(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    cfg = lib.Config(2048, 256, 8, 512, 512, 64, 16)
    assert L.moe_block_create(ctypes.byref(cfg), ctypes.byref(h)) == -6
    assert h.value is None


def test_binding_without_library_raises(tmp_path):
    saved = lib._LIB
    try:
        lib._LIB = None
        with pytest.raises(RuntimeError):
            lib.load_library(str(tmp_path / "missing.so"))
    finally:
        lib._LIB = saved


def test_stack_invalid_arguments_without_device(L):
    import torch
    h = ctypes.c_void_p()
    cfg = lib.Config(2048, 256, 8, 512, 512, 64, 1)
    assert L.moe_stack_create(None, 4, 1e-6, ctypes.byref(h)) == -1
    assert L.moe_stack_create(ctypes.byref(cfg), 0, 1e-6, ctypes.byref(h)) == -1
    assert L.moe_stack_create(ctypes.byref(cfg), 4, 0.0, ctypes.byref(h)) == -1
    assert L.moe_stack_create(ctypes.byref(cfg), 4, 1e-6, None) == -1
    bad = lib.Config(2048, 256, 8, 512, 512, 32, 1)
    assert L.moe_stack_create(ctypes.byref(bad), 4, 1e-6, ctypes.byref(h)) == -2
    if not torch.cuda.is_available():
        assert L.moe_stack_create(ctypes.byref(cfg), 4, 1e-6, ctypes.byref(h)) == -6
        assert h.value is None
    assert L.moe_stack_forward(None, None, None, 1, None, None) == -1
    assert L.moe_stack_load_layer(None, 0, None, 0, None) == -1
    assert L.moe_stack_get_status(None, None) == -1
    assert L.moe_stack_layer(None, 0) is None
