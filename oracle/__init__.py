"""CPU oracle for submanifold sparse convolution, K = 3 and 5 (test infrastructure).

Only the tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` may import this package.  The library's product path never
does: it shares no code, header or helper with the CUDA implementation.

The arithmetic lives in ``spconv_oracle.cpp`` (plain C++17: a hash-map
neighbour lookup, ``std::stable_sort`` for the mask order, and an fp64 sum over
the K^3 taps).  This module compiles it with the host C++ compiler and wraps it
with numpy arrays.  See the C++ file for the conventions and the passages each
function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spconv_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_DUPLICATE = -5
ERR_RANGE = -6


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (OpenMP if available)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = ["g++", "-std=c++17", "-O2", "-shared", "-fPIC", _SRC, "-o", tmp]
        try:
            subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True,
                           capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True, capture_output=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32 = ctypes.c_int64, ctypes.c_int32
        lib.oracle_kernel_map.argtypes = [P, i64, P, i32, i32, P]
        lib.oracle_kernel_map.restype = ctypes.c_int
        lib.oracle_masks.argtypes = [P, i64, i32, i32, i32, P]
        lib.oracle_masks.restype = None
        lib.oracle_tap_order.argtypes = [P, i64, i32, ctypes.c_int, P]
        lib.oracle_tap_order.restype = None
        lib.oracle_sort_keys.argtypes = [P, i64, i32, P, P]
        lib.oracle_sort_keys.restype = None
        lib.oracle_perm.argtypes = [P, i64, P]
        lib.oracle_perm.restype = None
        lib.oracle_pair_lists.argtypes = [P, P, i64, i32, i32, P, P, P]
        lib.oracle_pair_lists.restype = i64
        lib.oracle_conv_f64.argtypes = [P, i32, P, i64, P, P, i32, i32, P, i32]
        lib.oracle_conv_f64.restype = None
        lib.oracle_strided_map.argtypes = [P, i64, P, i32, P, P]
        lib.oracle_strided_map.restype = i64
        lib.oracle_inverse_map.argtypes = [P, i64, i64, P]
        lib.oracle_inverse_map.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__({ERR_DUPLICATE: "duplicate coordinate",
                          ERR_RANGE: "coordinate out of range"}.get(code, f"error {code}"))
        self.code = code


def kernel_map(coords, spatial_shape, batch_size: int, kernel_size: int = 3) -> np.ndarray:
    """``nbr[N, K^3]`` int32: row of the neighbour at tap k, or -1."""
    c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 4))
    shape = np.ascontiguousarray(np.asarray(spatial_shape, dtype=np.int32))
    K = int(kernel_size)
    assert K >= 1 and K % 2 == 1
    nbr = np.empty((c.shape[0], K ** 3), dtype=np.int32)
    rc = _load().oracle_kernel_map(_ptr(c), c.shape[0], _ptr(shape), int(batch_size), K, _ptr(nbr))
    if rc != 0:
        raise OracleError(rc)
    return nbr


def masks(nbr: np.ndarray, k0: int = 0, kg: int = None) -> np.ndarray:
    """Masks over the taps ``[k0, k0 + kg)`` (all taps when ``kg`` is None; at most 32)."""
    nbr = np.ascontiguousarray(nbr, dtype=np.int32)
    V = nbr.shape[1]
    kg = V - k0 if kg is None else int(kg)
    assert 0 < kg <= 32 and 0 <= k0 and k0 + kg <= V
    m = np.empty(nbr.shape[0], dtype=np.uint32)
    _load().oracle_masks(_ptr(nbr), nbr.shape[0], V, int(k0), kg, _ptr(m))
    return m


def tap_order(mask: np.ndarray, calibrated: bool = True, taps: int = 27) -> np.ndarray:
    """Key bit order of a group of ``taps`` taps (masks from ``masks``)."""
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    order = np.empty(int(taps), dtype=np.int32)
    _load().oracle_tap_order(_ptr(mask), mask.shape[0], int(taps), int(bool(calibrated)), _ptr(order))
    return order


def sort_keys(mask: np.ndarray, order: np.ndarray) -> np.ndarray:
    mask = np.ascontiguousarray(mask, dtype=np.uint32)
    order = np.ascontiguousarray(order, dtype=np.int32)
    key = np.empty(mask.shape[0], dtype=np.uint32)
    _load().oracle_sort_keys(_ptr(mask), mask.shape[0], order.shape[0], _ptr(order), _ptr(key))
    return key


def perm(key: np.ndarray) -> np.ndarray:
    key = np.ascontiguousarray(key, dtype=np.uint32)
    p = np.empty(key.shape[0], dtype=np.int32)
    _load().oracle_perm(_ptr(key), key.shape[0], _ptr(p))
    return p


def group_orders(nbr: np.ndarray, groups: int = 1, calibrated: bool = True):
    """Per group of ``V / groups`` consecutive taps: its masks, key bit order
    and row order (each group orders the rows by its own masks).  Returns
    ``(masks[G, N], orders[G, V/G], perms[G, N])``."""
    V = nbr.shape[1]
    assert V % groups == 0 and V // groups <= 32
    kg = V // groups
    ms, os_, ps = [], [], []
    for g in range(groups):
        m = masks(nbr, g * kg, kg)
        o = tap_order(m, calibrated, kg)
        ms.append(m)
        os_.append(o)
        ps.append(perm(sort_keys(m, o)))
    return np.stack(ms), np.stack(os_), np.stack(ps)


def pair_lists(nbr: np.ndarray, perm_: np.ndarray):
    """``(tap_off[V+1], in_rows[P], out_rows[P])``: the pairs of tap k in the
    row order of its group.  ``perm_`` is one order [N] (one group) or
    [G, N], one per group of V / G consecutive taps."""
    nbr = np.ascontiguousarray(nbr, dtype=np.int32)
    perm_ = np.ascontiguousarray(np.atleast_2d(perm_), dtype=np.int32)
    n, V = nbr.shape
    G = perm_.shape[0]
    assert V % G == 0 and perm_.shape[1] == n
    tap_off = np.empty(V + 1, dtype=np.int32)
    cap = max(1, V * n)
    ins = np.empty(cap, dtype=np.int32)
    outs = np.empty(cap, dtype=np.int32)
    p = _load().oracle_pair_lists(_ptr(nbr), _ptr(perm_), n, V, G, _ptr(tap_off), _ptr(ins), _ptr(outs))
    return tap_off, ins[:p].copy(), outs[:p].copy()


def conv_f64(nbr: np.ndarray, feats, weights, rows=None, threads: int = 0) -> np.ndarray:
    """fp64 ``out[r] = sum_k sum_c feats[nbr[r][k]][c] * weights[k][c][:]``.

    ``feats`` [N, C_in] and ``weights`` [V, C_in, C_out] (V = K^3, the width
    of ``nbr``) are taken as exact
    fp64 values (bf16 and fp32 inputs convert exactly).  ``rows`` selects the
    output rows to evaluate (all when None); the result follows its order.
    """
    nbr = np.ascontiguousarray(nbr, dtype=np.int32)
    f = np.ascontiguousarray(np.asarray(feats, dtype=np.float64))
    w = np.ascontiguousarray(np.asarray(weights, dtype=np.float64))
    c_in, c_out = int(w.shape[1]), int(w.shape[2])
    V = nbr.shape[1]
    assert w.shape[0] == V and f.shape[1] == c_in
    if rows is None:
        r_arr, n_rows, rp = None, nbr.shape[0], None
    else:
        r_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        n_rows, rp = r_arr.shape[0], _ptr(r_arr)
    out = np.empty((n_rows, c_out), dtype=np.float64)
    _load().oracle_conv_f64(_ptr(nbr), V, rp, n_rows, _ptr(f), _ptr(w), c_in, c_out, _ptr(out),
                            int(threads))
    return out


def strided_map(coords, spatial_shape, batch_size: int):
    """Strided convolution (kernel 3, stride 2, padding 1): ``(out_coords[M, 4], nbr[M, 27])``,
    the output sites in ascending (b, x, y, z) order and, per tap, the input row at 2o + d_k
    or -1 (see ``oracle_strided_map``)."""
    c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 4))
    shape = np.ascontiguousarray(np.asarray(spatial_shape, dtype=np.int32))
    cap = max(1, 8 * c.shape[0])
    oc = np.empty((cap, 4), dtype=np.int32)
    nbr = np.empty((cap, 27), dtype=np.int32)
    m = _load().oracle_strided_map(_ptr(c), c.shape[0], _ptr(shape), int(batch_size), _ptr(oc), _ptr(nbr))
    if m < 0:
        raise OracleError(int(m))
    return oc[:m].copy(), nbr[:m].copy()


def strided_shape(spatial_shape):
    """Output shape of the strided convolution: (X - 1) // 2 + 1 per axis."""
    return tuple((int(v) - 1) // 2 + 1 for v in spatial_shape)


def inverse_map(nbr: np.ndarray, n_in: int) -> np.ndarray:
    """The map of the inverse (transposed) convolution: ``inv[n_in, 27]``, the output site o
    of the strided map with 2o + d_k at input row i, or -1."""
    nbr = np.ascontiguousarray(nbr, dtype=np.int32)
    inv = np.empty((int(n_in), 27), dtype=np.int32)
    _load().oracle_inverse_map(_ptr(nbr), nbr.shape[0], int(n_in), _ptr(inv))
    return inv


def epilogue_f64(conv, scale=None, bias=None, residual=None, relu=False, rows=None) -> np.ndarray:
    """The layer epilogue on fp64 convolution sums ``conv`` [R, C_out]:
    ``y = conv * scale[o] + bias[o] + residual[row][o]``, then ``max(y, 0)``
    when ``relu`` -- a layer's inference-form batch norm (per-channel scale
    and shift), bias, residual branch and the ReLU that follows it ("Sparse
    convolution in FP32", "Offset-group partitioning": the ReLU applied to
    every output row; FlyDSL PR #942, "Open questions": layer stacks with
    normalisation and residuals).  ``residual`` is [N, C_out] in original row
    order; ``rows`` names the rows of ``conv`` (all N when None).  Missing
    terms are 1, 0 and 0.
    """
    y = np.array(conv, dtype=np.float64)
    if scale is not None:
        y = y * np.asarray(scale, dtype=np.float64)[None, :]
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    if residual is not None:
        r = np.asarray(residual, dtype=np.float64)
        y = y + (r if rows is None else r[np.asarray(rows)])
    if relu:
        y = np.maximum(y, 0.0)
    return y


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def subm_conv(coords, spatial_shape, batch_size, feats, weights, calibrated=True, rows=None,
              threads: int = 0, kernel_size: int = 3, groups: int = 1):
    """The whole path: kernel map, masks, order, pair lists and fp64 output.
    With one group, ``mask``/``order``/``perm`` are one array each; with
    ``groups`` > 1 they carry a leading group axis."""
    nbr = kernel_map(coords, spatial_shape, batch_size, kernel_size)
    m, order, p = group_orders(nbr, groups, calibrated)
    lists = pair_lists(nbr, p)
    out = conv_f64(nbr, feats, weights, rows=rows, threads=threads)
    if groups == 1:
        m, order, p = m[0], order[0], p[0]
    return dict(nbr=nbr, mask=m, order=order, perm=p, tap_off=lists[0], in_rows=lists[1],
                out_rows=lists[2], out=out)
