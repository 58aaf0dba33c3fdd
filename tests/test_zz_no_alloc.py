"""spconv_kernel_map_static: the kernel map without any device allocation.

Callers that cannot allocate device memory where they run (a plugin's
enqueue step in a runtime that plans all memory up front, a runtime that
forbids allocation after start-up) use this entry point; its working buffers
are a fixed file-scope device array.  Here it is called through the C ABI twice in a row
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


def test_static_map_at_the_row_limit_on_the_large_grid():
    """n = 65536 exactly (the scratch limit), two frames on the 2095 x 2095 x 695 grid whose
    dense volume overflows int32 (35-bit keys with the frame bit): bit for bit the allocating
    map, twice in a row."""
    build_mod.build()
    lib = _native.load()
    c, shape, _, _ = S.make_coords("large")
    c = c[:65536].copy()
    c[32768:, 0] = 1                            # the second half is frame 1
    coords = torch.from_numpy(c).cuda()
    ref = allocating_map(coords, shape, 2)
    assert (ref[:, :13] >= 0).any()             # the frames have neighbours, not only isolated voxels
    for _ in range(2):
        rc, nbr = static_map(lib, coords, shape, 2)
        assert rc == 0
        assert torch.equal(nbr, ref)


def test_static_map_63_bit_keys():
    """A (2^20 - 1)^3 grid: 21 bits per axis, 63 key bits, the widest key the sort takes.  A
    dense 12^3 block in the far corner (every top bit set) and scattered voxels."""
    build_mod.build()
    lib = _native.load()
    X = (1 << 20) - 1
    shape = (X, X, X)
    rng = np.random.default_rng(871)
    g = np.arange(X - 12, X)
    block = np.stack(np.meshgrid(g, g, g, indexing="ij"), -1).reshape(-1, 3)
    scatter = rng.integers(0, X, size=(500, 3))
    cells = np.unique(np.concatenate([block, scatter]), axis=0)
    c = np.concatenate([np.zeros((len(cells), 1), np.int64), cells], 1).astype(np.int32)
    c = c[rng.permutation(len(c))]
    coords = torch.from_numpy(c).cuda()
    ref = allocating_map(coords, shape, 1)
    rc, nbr = static_map(lib, coords, shape, 1)
    assert rc == 0
    assert torch.equal(nbr, ref)


def test_static_map_coordinate_out_of_range():
    """x = X (one past the last cell) is reported, not clamped or wrapped."""
    build_mod.build()
    lib = _native.load()
    c = torch.tensor([[0, 1, 1, 1], [0, 8, 2, 2], [0, 2, 2, 2]], dtype=torch.int32, device="cuda")
    rc, _ = static_map(lib, c, (8, 8, 8), 1)
    assert rc == -6
    rc, nbr = static_map(lib, c[:1].contiguous(), (8, 8, 8), 1)   # the status word was cleared again
    assert rc == 0
