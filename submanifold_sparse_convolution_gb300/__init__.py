"""GB300 (sm_103a) submanifold sparse 3x3x3 convolution.

A thin Python binding over the C ABI of ``libspconv.so`` (include/spconv.h):
the functions below only check and marshal arguments; every step of the path
(mapper, masks, sort, compaction, GEMM) runs in the library's CUDA kernels.
PyTorch supplies device memory and streams.

    m = build_map(coords)                       # int32 [N, 4] (b, x, y, z), CUDA
    out = subm_forward(m, feats, weights)       # bf16 [N, C_in] x [27, C_in, C_out]

One map serves every layer on the same sites; weights can be packed once, and
a layer's batch norm (inference form), bias, residual and ReLU are applied to
the fp32 sum before its single rounding:

    wp = wpack_create(weights)                  # [27 or 125, C_in, C_out]
    y = subm_forward_packed(m, x, wp, scale=s, bias=b, residual=x, relu=True)
    y32 = subm_forward(m, x.float(), weights.float())   # exact fp32 mode

Kernel size 5 and offset groups: ``build_map(coords, kernel_size=5)`` (125
taps, always five groups), ``build_map(coords, groups=3)``.  Downsampling and
its inverse, on the output sites of a stride-2 grid:

    d = build_map_strided(coords)               # sites o with a site in {2o + d}
    y = subm_forward(d, x, w)                   # [d.n, C_out] at map_out_coords(d)
    u = build_map_inverse(d)                    # back onto the input sites
    z = subm_forward(u, y, w2)                  # [N, C_out2]

Errors raise ``SpconvError`` with the library's status code; errors found on
the device (duplicate or out-of-range coordinates) surface through
``map_status`` or the next call on the map.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _native

__all__ = ["SpconvError", "Map", "WPack", "build_map", "subm_forward", "wpack_create",
           "subm_forward_packed", "map_status", "map_info", "map_export", "map_destroy",
           "last_launch_count", "status_string", "MAPPERS", "BIT_ORDERS", "PIPELINES", "GEMMS", "library"]

MAPPERS = {"auto": 0, "dense": 1, "sorted": 2, "hash": 3}
PIPELINES = {"auto": 0, "fused": 1, "multi": 2, "wide": 3}
GEMMS = {"auto": 0, "tile_union": 1, "tap_major": 2}
BIT_ORDERS = {"calibrated": 0, "plain": 1}
_DTYPES = {torch.bfloat16: 0, torch.float32: 1}


def library():
    """The loaded ctypes library (raises if it has not been built)."""
    return _native.load()


def status_string(code: int) -> str:
    """The library's message for a status code (``spconv_status_string``)."""
    return library().spconv_status_string(int(code)).decode()


class SpconvError(RuntimeError):
    """A call into the library returned a status other than SPCONV_OK; ``code`` holds it."""

    def __init__(self, code: int, where: str = ""):
        super().__init__(f"{where}: {status_string(code)} ({code})" if where else status_string(code))
        self.code = code


def _check(code: int, where: str):
    if code != 0:
        raise SpconvError(code, where)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _require_cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class Map:
    """A kernel map (handle ``spconv_map_t``); shared by every layer on these sites."""

    def __init__(self, handle: ctypes.c_void_p, n: int, coords: torch.Tensor, kernel_size: int = 3,
                 n_in: Optional[int] = None, keep=None):
        self._h = handle
        self.n = n                 # rows: the sites the output lives on
        self.n_in = n if n_in is None else n_in   # rows of the features a forward reads
        self.kernel_size = kernel_size
        self.taps = kernel_size ** 3
        self._coords = coords      # kept alive while the build may still read it
        self._keep = keep          # (an inverse map: the strided map it reads)

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise ValueError("map has been destroyed")
        return self._h

    def destroy(self):
        if getattr(self, "_h", None) is not None:
            library().spconv_map_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


class WPack:
    """Pre-packed weights (handle ``spconv_wpack_t``)."""

    def __init__(self, handle, c_in, c_out, dtype, src, taps=27):
        self._h = handle
        self.c_in, self.c_out, self.dtype, self.taps = c_in, c_out, dtype, taps
        self._src = src

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("weight pack has been destroyed")
        return self._h

    def destroy(self):
        if getattr(self, "_h", None) is not None:
            library().spconv_wpack_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def build_map(coords: torch.Tensor, spatial_shape: Optional[Sequence[int]] = None,
              batch_size: int = 0, kernel_size: int = 3, mapper: str = "auto",
              bit_order: str = "calibrated", dense_max_cells: int = 0, pipeline: str = "auto",
              gemm: str = "auto", stream: Optional[torch.cuda.Stream] = None, groups: int = 0) -> Map:
    """``spconv_build_map``: kernel map of ``coords`` (int32 [N, 4] (b, x, y, z) on the GPU).

    ``spatial_shape`` None and ``batch_size`` 0 derive them on the device
    (this synchronises the stream).  ``gemm`` picks the bf16 forward's work
    decomposition on this map (``GEMMS``).  ``kernel_size`` 3 or 5;
    ``groups`` the offset groups (0: 1 for K = 3, 5 for K = 5; or K).
    """
    lib = library()
    _require_cuda(coords, "coords")
    if coords.dtype != torch.int32 or coords.dim() != 2 or coords.shape[1] != 4:
        raise ValueError("coords must be int32 [N, 4]")
    shape_arr = None
    if spatial_shape is not None:
        shape_arr = (ctypes.c_int32 * 3)(*[int(v) for v in spatial_shape])
    opt = _native.Options(MAPPERS[mapper], BIT_ORDERS[bit_order], int(dense_max_cells),
                          PIPELINES[pipeline], GEMMS[gemm], int(groups))
    h = ctypes.c_void_p()
    rc = lib.spconv_build_map(_ptr(coords), int(coords.shape[0]),
                              ctypes.cast(shape_arr, _native.c_int32_p) if shape_arr is not None else None,
                              int(batch_size), int(kernel_size), ctypes.byref(opt), _stream_ptr(stream),
                              ctypes.byref(h))
    _check(rc, "spconv_build_map")
    return Map(h, int(coords.shape[0]), coords, int(kernel_size))


def _epilogue(n: int, c_out: int, dtype: torch.dtype, device, scale, bias, residual, relu):
    """The ``spconv_epilogue_t`` of a forward, or None when it is the identity.

    Returns (struct or None, tensors to keep alive until the call returns)."""
    if scale is None and bias is None and residual is None and not relu:
        return None, ()
    keep = []

    def vec(t, name):
        if t is None:
            return None
        _require_cuda(t, name)
        if t.dtype != torch.float32 or t.dim() != 1 or t.shape[0] != c_out or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 [{c_out}] tensor")
        keep.append(t)
        return t.data_ptr()

    e = _native.Epilogue()
    e.scale_dev = vec(scale, "scale")
    e.bias_dev = vec(bias, "bias")
    if residual is not None:
        _require_cuda(residual, "residual")
        if residual.dtype != dtype or tuple(residual.shape) != (n, c_out):
            raise ValueError(f"residual must be {dtype} [{n}, {c_out}]")
        keep.append(residual)
        e.residual_dev = residual.data_ptr()
    e.relu = 1 if relu else 0
    return e, tuple(keep)


def build_map_strided(coords: torch.Tensor, spatial_shape: Optional[Sequence[int]] = None,
                      batch_size: int = 0, kernel_size: int = 3, stride: int = 2, bit_order: str = "calibrated",
                      stream: Optional[torch.cuda.Stream] = None) -> Map:
    """``spconv_build_map_strided``: the map of a strided convolution (kernel 3, stride 2,
    padding 1) from the input sites ``coords``; its rows are the output sites
    (``map_out_coords``).  Synchronises the stream once."""
    lib = library()
    _require_cuda(coords, "coords")
    if coords.dtype != torch.int32 or coords.dim() != 2 or coords.shape[1] != 4:
        raise ValueError("coords must be int32 [N, 4]")
    shape_arr = None
    if spatial_shape is not None:
        shape_arr = (ctypes.c_int32 * 3)(*[int(v) for v in spatial_shape])
    opt = _native.Options(0, BIT_ORDERS[bit_order], 0, 0, 0, 0)
    h = ctypes.c_void_p()
    rc = lib.spconv_build_map_strided(_ptr(coords), int(coords.shape[0]),
                                      ctypes.cast(shape_arr, _native.c_int32_p) if shape_arr is not None else None,
                                      int(batch_size), int(kernel_size), int(stride), ctypes.byref(opt),
                                      _stream_ptr(stream), ctypes.byref(h))
    _check(rc, "spconv_build_map_strided")
    rows = ctypes.c_int64(0)
    _check(lib.spconv_map_rows(h, ctypes.byref(rows), None), "spconv_map_rows")   # (no second synchronisation)
    return Map(h, int(rows.value), coords, 3, n_in=int(coords.shape[0]))


def build_map_inverse(m: Map, bit_order: str = "calibrated") -> Map:
    """``spconv_build_map_inverse``: the map of the transposed convolution of strided map
    ``m``, from its output sites back onto its input sites."""
    opt = _native.Options(0, BIT_ORDERS[bit_order], 0, 0, 0, 0)
    h = ctypes.c_void_p()
    _check(library().spconv_build_map_inverse(m.handle, ctypes.byref(opt), ctypes.byref(h)),
           "spconv_build_map_inverse")
    return Map(h, m.n_in, m._coords, 3, n_in=m.n, keep=m)


def map_out_coords(m: Map, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """``spconv_map_out_coords``: a strided map's output sites, int32 [n, 4]."""
    out = torch.empty((m.n, 4), dtype=torch.int32, device=torch.device("cuda", torch.cuda.current_device()))
    _check(library().spconv_map_out_coords(m.handle, _ptr(out), _stream_ptr(stream)), "spconv_map_out_coords")
    return out


def subm_forward(m: Map, feats: torch.Tensor, weights: torch.Tensor,
                 out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None, *,
                 scale: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
                 residual: Optional[torch.Tensor] = None, relu: bool = False) -> torch.Tensor:
    """``spconv_subm_forward``: feats [N, C_in] x weights [V, C_in, C_out] -> [N, C_out], V = K^3.

    bf16 inputs use fp32 accumulation and one rounding at the store; fp32
    inputs take the exact fp32 path.  ``scale``/``bias`` (fp32 [C_out]),
    ``residual`` ([N, C_out], the output dtype; may be ``out``) and ``relu``
    are applied to each fp32 sum before that rounding
    (``spconv_subm_forward_ex``): y = sum*scale + bias + residual, then max(y, 0).
    """
    lib = library()
    _require_cuda(feats, "feats")
    _require_cuda(weights, "weights")
    if feats.dtype not in _DTYPES or weights.dtype != feats.dtype:
        raise ValueError("feats and weights must both be bf16 or both fp32")
    if feats.dim() != 2 or feats.shape[0] != m.n_in:
        raise ValueError(f"feats must be [{m.n_in}, C_in]")
    if weights.dim() != 3 or weights.shape[0] != m.taps or weights.shape[1] != feats.shape[1]:
        raise ValueError(f"weights must be [{m.taps}, C_in, C_out]")
    c_in, c_out = int(weights.shape[1]), int(weights.shape[2])
    if out is None:
        out = torch.empty((m.n, c_out), dtype=feats.dtype, device=feats.device)
    else:
        _require_cuda(out, "out")
        if out.dtype != feats.dtype or tuple(out.shape) != (m.n, c_out):
            raise ValueError(f"out must be {feats.dtype} [{m.n}, {c_out}]")
    epi, _keep = _epilogue(m.n, c_out, feats.dtype, feats.device, scale, bias, residual, relu)
    if epi is None:
        rc = lib.spconv_subm_forward(m.handle, _ptr(feats), _ptr(weights), _ptr(out), c_in, c_out,
                                     _DTYPES[feats.dtype], _stream_ptr(stream))
        _check(rc, "spconv_subm_forward")
    else:
        rc = lib.spconv_subm_forward_ex(m.handle, _ptr(feats), _ptr(weights), _ptr(out), c_in, c_out,
                                        _DTYPES[feats.dtype], ctypes.byref(epi), _stream_ptr(stream))
        _check(rc, "spconv_subm_forward_ex")
    return out


def wpack_create(weights: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> WPack:
    """``spconv_wpack_create_ex``: pack [K^3, C_in, C_out] weights (K = 3 or 5,
    from the first dimension) once for many forwards."""
    lib = library()
    _require_cuda(weights, "weights")
    sizes = {27: 3, 125: 5}
    if weights.dtype not in _DTYPES or weights.dim() != 3 or int(weights.shape[0]) not in sizes:
        raise ValueError("weights must be bf16 or fp32 [27 or 125, C_in, C_out]")
    c_in, c_out = int(weights.shape[1]), int(weights.shape[2])
    h = ctypes.c_void_p()
    rc = lib.spconv_wpack_create_ex(_ptr(weights), sizes[int(weights.shape[0])], c_in, c_out,
                                    _DTYPES[weights.dtype], _stream_ptr(stream), ctypes.byref(h))
    _check(rc, "spconv_wpack_create_ex")
    return WPack(h, c_in, c_out, weights.dtype, weights, int(weights.shape[0]))


def subm_forward_packed(m: Map, feats: torch.Tensor, wp: WPack, out: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None, *,
                        scale: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
                        residual: Optional[torch.Tensor] = None, relu: bool = False) -> torch.Tensor:
    """``spconv_subm_forward_packed``: forward with weights from ``wpack_create``;
    the epilogue arguments are those of ``subm_forward``."""
    lib = library()
    _require_cuda(feats, "feats")
    if feats.dtype != wp.dtype or feats.dim() != 2 or feats.shape != (m.n_in, wp.c_in):
        raise ValueError(f"feats must be {wp.dtype} [{m.n_in}, {wp.c_in}]")
    if wp.taps != m.taps:
        raise ValueError(f"weights pack has {wp.taps} taps, the map {m.taps}")
    if out is None:
        out = torch.empty((m.n, wp.c_out), dtype=feats.dtype, device=feats.device)
    else:
        _require_cuda(out, "out")
        if out.dtype != feats.dtype or tuple(out.shape) != (m.n, wp.c_out):
            raise ValueError(f"out must be {feats.dtype} [{m.n}, {wp.c_out}]")
    epi, _keep = _epilogue(m.n, wp.c_out, feats.dtype, feats.device, scale, bias, residual, relu)
    if epi is None:
        rc = lib.spconv_subm_forward_packed(m.handle, _ptr(feats), wp.handle, _ptr(out), _stream_ptr(stream))
        _check(rc, "spconv_subm_forward_packed")
    else:
        rc = lib.spconv_subm_forward_packed_ex(m.handle, _ptr(feats), wp.handle, _ptr(out), ctypes.byref(epi),
                                               _stream_ptr(stream))
        _check(rc, "spconv_subm_forward_packed_ex")
    return out


def subm_forward_layers(m: Map, feats: torch.Tensor, wps: Sequence[WPack], relu: Sequence[bool] = (),
                        outs: Optional[Sequence[torch.Tensor]] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> list:
    """``spconv_subm_forward_layers``: ``len(wps)`` layers over map ``m`` in one launch;
    layer l reads layer l - 1's output (layer 0: ``feats``) and applies a ReLU
    when ``relu[l]``.  ``outs`` gives one output per layer (consecutive ones may
    not overlap; two buffers may alternate); by default two buffers alternate.
    Returns the list of per-layer outputs (views of ``outs``)."""
    lib = library()
    _require_cuda(feats, "feats")
    L = len(wps)
    if L < 1:
        raise ValueError("at least one layer")
    wp0 = wps[0]
    if feats.dtype != torch.bfloat16 or tuple(feats.shape) != (m.n_in, wp0.c_in):
        raise ValueError(f"feats must be bf16 [{m.n_in}, {wp0.c_in}]")
    relu = list(relu) + [False] * (L - len(relu))
    if outs is None:
        bufs = [torch.empty((m.n, wp0.c_out), dtype=feats.dtype, device=feats.device) for _ in range(min(L, 2))]
        outs = [bufs[l % 2] for l in range(L)]
    else:
        outs = list(outs)
        if len(outs) != L:
            raise ValueError(f"{L} outputs expected")
        for o in outs:
            _require_cuda(o, "out")
            if o.dtype != feats.dtype or tuple(o.shape) != (m.n, wp0.c_out):
                raise ValueError(f"outputs must be bf16 [{m.n}, {wp0.c_out}]")
    wh = (ctypes.c_void_p * L)(*[w.handle for w in wps])
    oh = (ctypes.c_void_p * L)(*[_ptr(o) for o in outs])
    epis = (_native.Epilogue * L)()
    for l in range(L):
        epis[l].relu = 1 if relu[l] else 0
    rc = lib.spconv_subm_forward_layers(m.handle, _ptr(feats), ctypes.cast(wh, ctypes.POINTER(ctypes.c_void_p)),
                                        ctypes.cast(oh, ctypes.POINTER(ctypes.c_void_p)), L, epis,
                                        _stream_ptr(stream))
    _check(rc, "spconv_subm_forward_layers")
    return outs


def map_status(m: Map) -> int:
    """``spconv_map_status``: 0, or the first device-detected error code (synchronises)."""
    return int(library().spconv_map_status(m.handle))


def map_info(m: Map) -> dict:
    """``spconv_map_info`` as a dict (synchronises)."""
    info = _native.MapInfo()
    _check(library().spconv_map_info(m.handle, ctypes.byref(info)), "spconv_map_info")
    return dict(n=info.n, pairs=info.pairs, n_tiles=info.n_tiles, tile_taps=info.tile_taps,
                mapper={1: "dense", 2: "sorted", 3: "hash"}.get(info.mapper, str(info.mapper)),
                pipeline={1: "fused", 2: "multi", 3: "wide"}.get(info.pipeline, str(info.pipeline)),
                key_bits=info.key_bits, shape=tuple(info.shape), batch_size=info.batch_size,
                gemm={1: "tile_union", 2: "tap_major"}.get(info.gemm, str(info.gemm)),
                kernel_size=info.kernel_size, groups=info.groups, n_in=info.n_in,
                conv={0: "submanifold", 1: "strided", 2: "inverse"}.get(info.conv, str(info.conv)),
                out_shape=tuple(info.out_shape))


def map_export(m: Map, stream: Optional[torch.cuda.Stream] = None) -> dict:
    """``spconv_map_export``: nbr [N, V], tap_off [V+1], in_rows/out_rows [P];
    mask and perm [N] with one offset group, [G, N] with G > 1."""
    info = map_info(m)
    n, p = info["n"], info["pairs"]
    V, G = info["kernel_size"] ** 3, info["groups"]
    dev = torch.device("cuda", torch.cuda.current_device())
    nbr = torch.empty((n, V), dtype=torch.int32, device=dev)
    gshape = (n,) if G == 1 else (G, n)
    mask = torch.empty(gshape, dtype=torch.int32, device=dev)
    perm = torch.empty(gshape, dtype=torch.int32, device=dev)
    tap_off = torch.empty((V + 1,), dtype=torch.int32, device=dev)
    ins = torch.empty((max(p, 1),), dtype=torch.int32, device=dev)
    outs = torch.empty((max(p, 1),), dtype=torch.int32, device=dev)
    rc = library().spconv_map_export(m.handle, _ptr(nbr), _ptr(mask), _ptr(perm), _ptr(tap_off),
                                     _ptr(ins), _ptr(outs), _stream_ptr(stream))
    _check(rc, "spconv_map_export")
    return dict(nbr=nbr, mask=mask, perm=perm, tap_off=tap_off, in_rows=ins[:p], out_rows=outs[:p],
                info=info)


def map_destroy(m: Map):
    """``spconv_map_destroy``."""
    m.destroy()


def last_launch_count() -> int:
    """Kernels the library launched in its last call on this thread."""
    return int(library().spconv_last_launch_count())
