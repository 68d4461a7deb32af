"""The C-ABI library loads and exports every entry point its header declares; host-side
argument checks that need no GPU."""
import ctypes
import os
import re

import pytest

import sparse_moe_layer_15_b300 as fm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(flint_(?:moe|dense|swa)_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert set(declared_functions()) == set(fm.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = fm.load_library()
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    lib = fm.load_library()
    for code in range(7):
        s = lib.flint_moe_status_string(code)
        assert s and s != b"unknown status"
    assert lib.flint_moe_status_string(99) == b"unknown status"


def test_workspace_bytes_and_shape_refusal():
    n = fm.workspace_bytes(16)
    assert n > 0 and n % 256 == 0
    assert fm.workspace_bytes(256) > n
    lib = fm.load_library()
    bad = fm._Config(4096, 256, 6, 512, 1024, 16, 0, 1e-6)
    out = ctypes.c_size_t(0)
    assert lib.flint_moe_workspace_bytes(ctypes.byref(bad), ctypes.byref(out)) == 2  # unsupported
    bad = fm._Config(2048, 256, 8, 512, 1024, 16, 0, 1e-6)
    assert lib.flint_moe_workspace_bytes(ctypes.byref(bad), ctypes.byref(out)) == 2
    zero = fm._Config(2048, 256, 6, 512, 1024, 0, 0, 1e-6)
    assert lib.flint_moe_workspace_bytes(ctypes.byref(zero), ctypes.byref(out)) == 1  # invalid
    prenorm_no_eps = fm._Config(2048, 256, 6, 512, 1024, 16, fm.FLAG_PRE_RMSNORM, 0.0)
    assert lib.flint_moe_workspace_bytes(ctypes.byref(prenorm_no_eps), ctypes.byref(out)) == 1
    unknown_flag = fm._Config(2048, 256, 6, 512, 1024, 16, 0x100, 1e-6)
    assert lib.flint_moe_workspace_bytes(ctypes.byref(unknown_flag), ctypes.byref(out)) == 2


def test_null_handle_calls_are_rejected():
    lib = fm.load_library()
    assert lib.flint_moe_forward(None, None, 1, None, None, None, None) == 1
    assert lib.flint_moe_route(None, None, 1, None, None, None, None) == 1
    assert lib.flint_moe_destroy(None) == 1
    assert lib.flint_moe_poll_device_status(None, None) == 1


def test_create_rejects_missing_workspace_before_touching_a_device():
    lib = fm.load_library()
    cfg = fm._Config(2048, 256, 6, 512, 1024, 16, 0, 1e-6)
    w = fm._Weights(*([256] * 8))  # aligned dummies, never dereferenced
    h = ctypes.c_void_p()
    assert lib.flint_moe_create(ctypes.byref(cfg), ctypes.byref(w), None, 0, ctypes.byref(h)) == 3
    w_bad = fm._Weights(*([258] * 8))  # misaligned
    assert lib.flint_moe_create(ctypes.byref(cfg), ctypes.byref(w_bad), None, 0, ctypes.byref(h)) == 1


def test_stack_workspace_and_argument_checks():
    lib = fm.load_library()
    flags = fm.FLAG_PRE_RMSNORM | fm.FLAG_RESIDUAL
    one = fm.stack_workspace_bytes(1, 256, flags)
    many = fm.stack_workspace_bytes(47, 256, flags)
    assert one % 256 == 0 and many > one and many - one < 47 * 2048  # a table entry per layer
    cfg = fm._Config(2048, 256, 6, 512, 1024, 256, flags, 1e-6)
    out = ctypes.c_size_t(0)
    assert lib.flint_moe_stack_workspace_bytes(ctypes.byref(cfg), 0, ctypes.byref(out)) == 1  # no layers
    big = fm._Config(2048, 256, 6, 512, 1024, 512, flags, 1e-6)
    assert lib.flint_moe_stack_workspace_bytes(ctypes.byref(big), 4, ctypes.byref(out)) == 2  # decode sizes only
    arr = (fm._Weights * 2)(fm._Weights(*([256] * 8)), fm._Weights(*([256] * 8)))
    h = ctypes.c_void_p()
    assert lib.flint_moe_stack_create(ctypes.byref(cfg), arr, 2, None, 0, ctypes.byref(h)) == 3
    arr[1] = fm._Weights(*([258] * 8))  # misaligned second layer
    assert lib.flint_moe_stack_create(ctypes.byref(cfg), arr, 2, ctypes.c_void_p(256), 1 << 40,
                                      ctypes.byref(h)) == 1
    assert lib.flint_moe_stack_forward(None, None, 1, None, None, None) == 1
    assert lib.flint_moe_stack_poll_device_status(None, None) == 1
    assert lib.flint_moe_stack_destroy(None) == 1
