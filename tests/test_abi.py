"""The C-ABI library builds for sm_103a, loads, and exports what include/spconv.h declares.

No call here launches device work: only argument checks that return before
any CUDA call are exercised.
"""
import ctypes
import os
import re

import pytest

from submanifold_sparse_convolution_gb300 import _native
from submanifold_sparse_convolution_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _native.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "spconv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spconv_[a-z_]+)\s*\(", src)))


def test_header_declares_the_path():
    names = declared_functions()
    for required in ("spconv_build_map", "spconv_subm_forward", "spconv_map_destroy",
                     "spconv_map_status", "spconv_map_export", "spconv_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(_native.SIGNATURES)


def test_status_strings(lib):
    for code, text in [(0, "ok"), (-1, "invalid argument"), (-5, "duplicate coordinate"),
                       (-6, "coordinate out of range"), (-7, "output overlaps input"),
                       (-8, "kernel wait timed out"), (-9, "internal consistency check failed"),
                       (-99, "unknown status")]:
        assert lib.spconv_status_string(code).decode() == text


def test_host_side_argument_errors(lib):
    h = ctypes.c_void_p()
    shape = (ctypes.c_int32 * 3)(4, 4, 4)
    sp = ctypes.cast(shape, _native.c_int32_p)
    # null output handle
    assert lib.spconv_build_map(None, 0, sp, 1, 3, None, None, None) == -1
    # negative n, oversize n
    assert lib.spconv_build_map(None, -1, sp, 1, 3, None, None, ctypes.byref(h)) == -1
    assert lib.spconv_build_map(None, 1 << 30, sp, 1, 3, None, None, ctypes.byref(h)) == -1
    # n > 0 with null or misaligned coordinates
    assert lib.spconv_build_map(None, 5, sp, 1, 3, None, None, ctypes.byref(h)) == -1
    assert lib.spconv_build_map(ctypes.c_void_p(8), 5, sp, 1, 3, None, None, ctypes.byref(h)) == -1
    # kernel sizes other than 3 and 5
    for k in (1, 2, 4, 7):
        assert lib.spconv_build_map(None, 0, sp, 1, k, None, None, ctypes.byref(h)) == -2
    # bad options
    for bad in [(7, 0, 0, 0, 0), (0, 3, 0, 0, 0), (0, 0, -1, 0, 0), (0, 0, 0, 4, 0), (0, 0, 0, 0, 3),
                (0, 0, 0, 0, -1), (0, 0, 0, 0, 0, -1)]:
        opt = _native.Options(*bad)
        assert lib.spconv_build_map(None, 0, sp, 1, 3, ctypes.byref(opt), None, ctypes.byref(h)) == -1
    # offset groups: 1 or K; more than one only with the MULTI pipeline and the TILE_UNION forward
    for k, extra in [(3, (0, 0, 0, 0, 0, 2)), (5, (0, 0, 0, 0, 0, 1)), (5, (0, 0, 0, 3, 0, 0)),
                     (5, (0, 0, 0, 1, 0, 5)), (3, (0, 0, 0, 0, 2, 3))]:
        opt = _native.Options(*extra)
        assert lib.spconv_build_map(None, 0, sp, 1, k, ctypes.byref(opt), None, ctypes.byref(h)) == -2
    assert lib.spconv_wpack_create_ex(None, 5, 16, 16, 0, None, ctypes.byref(h)) == -1
    assert lib.spconv_wpack_create_ex(ctypes.c_void_p(256), 7, 16, 16, 0, None, ctypes.byref(h)) == -2
    # null handles everywhere else
    assert lib.spconv_subm_forward(None, None, None, None, 16, 16, 0, None) == -1
    assert lib.spconv_subm_forward_packed(None, None, None, None, None) == -1
    assert lib.spconv_wpack_create(None, 16, 16, 0, None, ctypes.byref(h)) == -1
    assert lib.spconv_map_status(None) == -1
    info = _native.MapInfo()
    assert lib.spconv_map_info(None, ctypes.byref(info)) == -1
    assert lib.spconv_map_rows(None, None, None) == -1
    assert lib.spconv_map_export(None, None, None, None, None, None, None, None) == -1
    lib.spconv_map_destroy(None)
    lib.spconv_wpack_destroy(None)
    assert lib.spconv_last_launch_count() == 0


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="build the CUDA library"):
        _native.open_library(str(tmp_path / "missing.so"))


def test_library_is_built_for_sm103a():
    flags = build_mod.NVCC_FLAGS
    assert "arch=compute_103a,code=sm_103a" in flags
