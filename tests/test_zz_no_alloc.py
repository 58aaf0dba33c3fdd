"""spconv_kernel_map_static: the kernel map without any device allocation.

Callers that cannot allocate device memory where they run (a plugin's
enqueue step in a runtime that plans all memory up front, code running while
its stream is captured) use this entry point; its working buffers are a fixed
file-scope device array.  Here it is called through the C ABI twice in a row
and must reproduce, bit for bit, the kernel map that the allocating entry
point (spconv_build_map + spconv_map_export) gives for the same coordinates.
This file is collected last so that a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest
import torch

import submanifold_sparse_convolution_gb300 as sc
from submanifold_sparse_convolution_gb300 import _native
from submanifold_sparse_convolution_gb300 import build as build_mod
from submanifold_sparse_convolution_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def static_map(lib, coords, shape, batch):
    n = coords.shape[0]
    nbr = torch.full((n, 27), -7, dtype=torch.int32, device="cuda")
    sh = (ctypes.c_int32 * 3)(*shape)
    rc = lib.spconv_kernel_map_static(ctypes.c_void_p(coords.data_ptr()), n, ctypes.cast(sh, _native.c_int32_p),
                                      batch, ctypes.c_void_p(nbr.data_ptr()),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, nbr


def allocating_map(coords, shape, batch):
    return sc.map_export(sc.build_map(coords, shape, batch))["nbr"]


def test_static_map_matches_allocating_map_twice():
    build_mod.build()
    lib = _native.load()
    cases = [S.make_coords("tiny")[:3], S.random_cloud(5, 60000, shape=(64, 64, 64), batch_size=3)]
    for case in cases:
        if isinstance(case, tuple):
            c, shape, batch = case
            coords = torch.from_numpy(c).cuda()
        else:
            coords, shape, batch = case.coords.cuda(), case.spatial_shape, case.batch_size
        ref = allocating_map(coords, shape, batch)
        for _ in range(2):                    # the shared scratch keeps the previous call's contents
            rc, nbr = static_map(lib, coords, shape, batch)
            assert rc == 0
            assert torch.equal(nbr, ref)


def test_static_map_limits_and_errors():
    build_mod.build()
    lib = _native.load()
    big = torch.zeros((65537, 4), dtype=torch.int32, device="cuda")
    rc, _ = static_map(lib, big, (8, 8, 8), 1)
    assert rc == -1                            # beyond the fixed scratch: rejected, nothing launched
    dup = torch.tensor([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=torch.int32, device="cuda")
    rc, _ = static_map(lib, dup, (4, 4, 4), 1)
    assert rc == -5
    rc, nbr = static_map(lib, torch.tensor([[0, 3, 3, 3]], dtype=torch.int32, device="cuda"), (8, 8, 8), 1)
    assert rc == 0 and nbr.cpu().numpy()[0].tolist() == [-1] * 13 + [0] + [-1] * 13
