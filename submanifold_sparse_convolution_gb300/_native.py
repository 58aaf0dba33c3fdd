"""ctypes declarations of libspconv's C ABI (include/spconv.h).

Loading fails loudly when the library has not been built: there is no CPU or
PyTorch fallback for any step of the path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libspconv.so")

c_int32_p = ctypes.POINTER(ctypes.c_int32)


class Options(ctypes.Structure):
    _fields_ = [("mapper", ctypes.c_int32), ("bit_order", ctypes.c_int32),
                ("dense_max_cells", ctypes.c_int64), ("pipeline", ctypes.c_int32),
                ("gemm", ctypes.c_int32), ("groups", ctypes.c_int32)]


class MapInfo(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("pairs", ctypes.c_int64), ("n_tiles", ctypes.c_int64),
                ("tile_taps", ctypes.c_int64), ("mapper", ctypes.c_int32),
                ("pipeline", ctypes.c_int32),
                ("key_bits", ctypes.c_int32), ("shape", ctypes.c_int32 * 3),
                ("batch_size", ctypes.c_int32), ("gemm", ctypes.c_int32),
                ("kernel_size", ctypes.c_int32), ("groups", ctypes.c_int32),
                ("n_in", ctypes.c_int64), ("conv", ctypes.c_int32), ("out_shape", ctypes.c_int32 * 3)]


class Epilogue(ctypes.Structure):
    _fields_ = [("scale_dev", ctypes.c_void_p), ("bias_dev", ctypes.c_void_p),
                ("residual_dev", ctypes.c_void_p), ("relu", ctypes.c_int32)]


# name -> (restype, argtypes)
SIGNATURES = {
    "spconv_build_map": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, c_int32_p, ctypes.c_int32,
                                        ctypes.c_int32, ctypes.POINTER(Options), ctypes.c_void_p,
                                        ctypes.POINTER(ctypes.c_void_p)]),
    "spconv_build_map_strided": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, c_int32_p, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(Options),
                                                ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    "spconv_build_map_inverse": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(Options),
                                                ctypes.POINTER(ctypes.c_void_p)]),
    "spconv_map_out_coords": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "spconv_subm_forward": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_void_p]),
    "spconv_subm_forward_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.POINTER(Epilogue),
                                              ctypes.c_void_p]),
    "spconv_wpack_create": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_void_p,
                                           ctypes.POINTER(ctypes.c_void_p)]),
    "spconv_wpack_create_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                                              ctypes.POINTER(ctypes.c_void_p)]),
    "spconv_subm_forward_packed": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_void_p]),
    "spconv_subm_forward_packed_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.POINTER(Epilogue),
                                                     ctypes.c_void_p]),
    "spconv_wpack_destroy": (None, [ctypes.c_void_p]),
    "spconv_subm_forward_layers": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p),
                                                  ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32,
                                                  ctypes.POINTER(Epilogue), ctypes.c_void_p]),
    "spconv_map_status": (ctypes.c_int, [ctypes.c_void_p]),
    "spconv_map_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(MapInfo)]),
    "spconv_map_rows": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "spconv_map_export": (ctypes.c_int, [ctypes.c_void_p] + [ctypes.c_void_p] * 6 + [ctypes.c_void_p]),
    "spconv_map_destroy": (None, [ctypes.c_void_p]),
    "spconv_kernel_map_static": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, c_int32_p, ctypes.c_int32,
                                                ctypes.c_void_p, ctypes.c_void_p]),
    "spconv_last_launch_count": (ctypes.c_int32, []),
    "spconv_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]),
    "spconv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def open_library(path: str):
    """Open a libspconv build at ``path`` and declare its functions."""
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m submanifold_sparse_convolution_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load():
    """The in-tree libspconv.so, opened once per process."""
    global _lib
    if _lib is None:
        _lib = open_library(LIB_PATH)
    return _lib
