"""Seeded synthetic voxel clouds, features and weights.

This module only draws inputs.  It holds none of the convolution's arithmetic
(no neighbour search, no sums): the same arrays feed the CUDA library and the
CPU oracle, and neither side imports the other.

The workloads stand in for the LiDAR and indoor scans that the pages measure
on (nuScenes, SemanticKITTI, ScanNet are not available here).  They follow the
shapes the pages give: ground-plane voxel sets plus object surfaces, row order
uncorrelated with space, features ~N(0,1) and weights ~N(0, 1/sqrt(27*C_in))
rounded to bf16.

Coordinates are ``int32 [N, 4]`` rows ``(b, x, y, z)``; every row is unique.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Tuple

import numpy as np
import torch

BASE_SEED = 20261202


@dataclasses.dataclass
class Workload:
    name: str
    coords: torch.Tensor            # int32 [N, 4] (b, x, y, z), CPU
    spatial_shape: Tuple[int, int, int]
    batch_size: int
    c_in: int
    c_out: int
    feats: torch.Tensor             # bf16 [N, C_in], CPU
    weights: List[torch.Tensor]     # per layer bf16 [27, C_in, C_out], CPU
    seed: int

    @property
    def n(self) -> int:
        return int(self.coords.shape[0])

    @property
    def layers(self) -> int:
        return len(self.weights)


# ---------------------------------------------------------------------------
# coordinate sets
# ---------------------------------------------------------------------------

def uniform_cells(rng: np.random.Generator, n: int, shape: Tuple[int, int, int],
                  batch: int = 0) -> np.ndarray:
    """``n`` distinct cells drawn uniformly without replacement from ``shape``."""
    X, Y, Z = shape
    lin = rng.choice(X * Y * Z, size=n, replace=False)
    x = lin // (Y * Z)
    y = (lin // Z) % Y
    z = lin % Z
    b = np.full(n, batch, dtype=np.int64)
    return np.stack([b, x, y, z], axis=1).astype(np.int32)


def _ground_rings(rng, shape, radius, z_base, n_rings, r_min):
    """LiDAR-like ground returns: concentric scan rings about the grid centre.

    Ring ``j`` sits at radius ``r_min * (radius / r_min) ** (j / (n_rings - 1))``
    (geometric spacing, as beams at fixed elevation steps meet flat ground) and
    is the digital circle of cells within half a cell of it.  The ground height
    along a ring is ``z0 = z_base + e`` with a jitter ``e`` in {-1, 0, +1} that
    is constant over random arcs of 8..64 cells; each return occupies the two
    layers ``z0`` and ``z0 + 1``.
    """
    X, Y, Z = shape
    cx, cy = (X - 1) / 2.0, (Y - 1) / 2.0
    pts = []
    for j in range(n_rings):
        r = r_min * (radius / r_min) ** (j / max(1, n_rings - 1))
        m = int(np.ceil(r)) + 1
        gx, gy = np.meshgrid(np.arange(int(cx) - m, int(cx) + m + 2),
                             np.arange(int(cy) - m, int(cy) + m + 2), indexing="ij")
        d = np.sqrt((gx - cx) ** 2 + (gy - cy) ** 2)
        on = np.abs(d - r) < 0.5
        gx, gy = gx[on], gy[on]
        ang = np.arctan2(gy - cy, gx - cx)
        order = np.argsort(ang, kind="stable")
        gx, gy = gx[order], gy[order]
        jit = np.empty(gx.shape[0], dtype=np.int64)
        i = 0
        while i < gx.shape[0]:
            run = int(rng.integers(8, 65))
            jit[i:i + run] = rng.integers(-1, 2)
            i += run
        z0 = z_base + jit
        pts.append(np.stack([gx, gy, z0], 1))
        pts.append(np.stack([gx, gy, z0 + 1], 1))
    return np.concatenate(pts, 0)


def _box_surface(x0, y0, z0, sx, sy, sz):
    """Cells on the six faces of the box [x0,x0+sx) x [y0,y0+sy) x [z0,z0+sz)."""
    gx, gy, gz = np.meshgrid(np.arange(x0, x0 + sx), np.arange(y0, y0 + sy),
                             np.arange(z0, z0 + sz), indexing="ij")
    face = ((gx == x0) | (gx == x0 + sx - 1) | (gy == y0) | (gy == y0 + sy - 1)
            | (gz == z0) | (gz == z0 + sz - 1))
    return np.stack([gx[face], gy[face], gz[face]], 1)


def _cylinder_surface(cx, cy, z0, radius, height):
    """Cells within half a cell of a vertical cylinder's side, plus its top disc."""
    r = int(np.ceil(radius)) + 1
    gx, gy = np.meshgrid(np.arange(cx - r, cx + r + 1), np.arange(cy - r, cy + r + 1),
                         indexing="ij")
    d = np.sqrt((gx - cx) ** 2 + (gy - cy) ** 2)
    ring = np.abs(d - radius) < 0.5
    top = d <= radius
    parts = []
    for z in range(z0, z0 + height):
        parts.append(np.stack([gx[ring], gy[ring], np.full(ring.sum(), z)], 1))
    parts.append(np.stack([gx[top], gy[top], np.full(top.sum(), z0 + height - 1)], 1))
    return np.concatenate(parts, 0)


def surface_cells(rng: np.random.Generator, n: int, shape: Tuple[int, int, int], *,
                  radius: float, z_base: int, n_rings: int, r_min: float, n_boxes: int,
                  box_side=(3, 12), box_height=(3, 10), n_cylinders: int = 0,
                  cyl_radius=(2, 8), isolated_frac: float = 0.0, batch: int = 0) -> np.ndarray:
    """A LiDAR-like set of exactly ``n`` unique cells.

    Candidates: ``n_rings`` jittered two-layer ground scan rings out to
    ``radius`` about the grid centre, ``n_boxes`` axis-aligned box surfaces and
    ``n_cylinders`` vertical cylinder surfaces standing on the ground inside
    that disc.  The candidates
    are subsampled without replacement to ``n - n_isolated`` cells, then
    ``n_isolated = round(isolated_frac * n)`` cells uniform over the whole grid
    are added (redrawn until every cell is unique).
    """
    X, Y, Z = shape
    cand = [_ground_rings(rng, shape, radius, z_base, n_rings, r_min)]
    cx, cy = (X - 1) / 2.0, (Y - 1) / 2.0
    for _ in range(n_boxes):
        a = rng.uniform(0, 2 * np.pi)
        rr = radius * np.sqrt(rng.uniform(0, 1))
        sx = int(rng.integers(box_side[0], box_side[1] + 1))
        sy = int(rng.integers(box_side[0], box_side[1] + 1))
        sz = int(rng.integers(box_height[0], box_height[1] + 1))
        x0 = int(cx + rr * np.cos(a)) - sx // 2
        y0 = int(cy + rr * np.sin(a)) - sy // 2
        cand.append(_box_surface(x0, y0, z_base, sx, sy, sz))
    for _ in range(n_cylinders):
        a = rng.uniform(0, 2 * np.pi)
        rr = radius * np.sqrt(rng.uniform(0, 1))
        rad = float(rng.uniform(cyl_radius[0], cyl_radius[1]))
        h = int(rng.integers(box_height[0], box_height[1] + 1))
        cand.append(_cylinder_surface(int(cx + rr * np.cos(a)), int(cy + rr * np.sin(a)),
                                      z_base, rad, h))
    pts = np.concatenate(cand, 0).astype(np.int64)
    ok = ((pts[:, 0] >= 0) & (pts[:, 0] < X) & (pts[:, 1] >= 0) & (pts[:, 1] < Y)
          & (pts[:, 2] >= 0) & (pts[:, 2] < Z))
    pts = pts[ok]
    lin = np.unique((pts[:, 0] * Y + pts[:, 1]) * Z + pts[:, 2])
    n_iso = int(round(isolated_frac * n))
    n_surf = n - n_iso
    if lin.shape[0] < n_surf:
        raise ValueError(f"surface generator made {lin.shape[0]} cells, need {n_surf}")
    lin = rng.choice(lin, size=n_surf, replace=False)
    if n_iso:
        taken = set(lin.tolist())
        extra = []
        while len(extra) < n_iso:
            c = int(rng.integers(0, X * Y * Z))
            if c not in taken:
                taken.add(c)
                extra.append(c)
        lin = np.concatenate([lin, np.array(extra, dtype=np.int64)])
    x = lin // (Y * Z)
    y = (lin // Z) % Y
    z = lin % Z
    b = np.full(n, batch, dtype=np.int64)
    return np.stack([b, x, y, z], 1).astype(np.int32)


def shuffle_rows(rng: np.random.Generator, coords: np.ndarray) -> np.ndarray:
    return coords[rng.permutation(coords.shape[0])]


# ---------------------------------------------------------------------------
# features and weights
# ---------------------------------------------------------------------------

def bf16_normal(rng: np.random.Generator, shape, std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) drawn in float64, rounded to bf16 (round to nearest even)."""
    x = rng.standard_normal(size=shape) * std
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)


def weights_std(c_in: int, taps: int = 27) -> float:
    return 1.0 / float(np.sqrt(float(taps) * c_in))


def make_weights(rng, c_in, c_out, taps: int = 27) -> torch.Tensor:
    """``[taps, C_in, C_out]`` bf16, std 1/sqrt(taps*C_in) (fan-in scaling)."""
    return bf16_normal(rng, (taps, c_in, c_out), weights_std(c_in, taps))


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

#: name -> (index, description)
CONFIG_NAMES = ["tiny", "outdoor", "deep", "large", "stage"]

# Generator parameters, chosen offline so that the mean number of present taps
# per voxel (centre tap included) is about 7 on the outdoor-like clouds (the
# deep, compact stage comes out denser, about 8).
_OUTDOOR = dict(radius=170.0, n_rings=40, r_min=8.0, z_base=8, n_boxes=60)
_DEEP = dict(radius=80.0, n_rings=50, r_min=3.0, z_base=8, n_boxes=60, box_side=(2, 6),
             box_height=(3, 10))
_LARGE = dict(radius=330.0, n_rings=70, r_min=8.0, z_base=20, n_boxes=75, n_cylinders=75,
              isolated_frac=0.05)
_STAGE = dict(radius=420.0, n_rings=95, r_min=8.0, z_base=8, n_boxes=60)


def make_coords(name: str, seed: Optional[int] = None):
    """Coordinates, spatial shape and batch size of workload ``name``."""
    idx = CONFIG_NAMES.index(name)
    seed = BASE_SEED + idx + 1 if seed is None else seed
    rng = np.random.default_rng(seed)
    if name == "tiny":
        shape = (32, 32, 32)
        c = uniform_cells(rng, 2000, shape)
        return shuffle_rows(rng, c), shape, 1, rng
    if name == "outdoor":
        shape = (1440, 1440, 40)
        c = surface_cells(rng, 32371, shape, **_OUTDOOR)
        return shuffle_rows(rng, c), shape, 1, rng
    if name == "deep":
        shape = (180, 180, 41)
        c = surface_cells(rng, 15052, shape, **_DEEP)
        return shuffle_rows(rng, c), shape, 1, rng
    if name == "large":
        shape = (2095, 2095, 695)
        c = surface_cells(rng, 94517, shape, **_LARGE)
        return shuffle_rows(rng, c), shape, 1, rng
    if name == "stage":
        shape = (1440, 1440, 40)
        frames = [surface_cells(rng, 120000, shape, batch=b, **_STAGE) for b in range(2)]
        return shuffle_rows(rng, np.concatenate(frames, 0)), shape, 2, rng
    raise KeyError(name)


_CHANNELS = {"tiny": (16, 16, 1), "outdoor": (128, 128, 1), "deep": (512, 512, 1),
             "large": (128, 128, 1), "stage": (64, 64, 6)}


def make_workload(name: str, seed: Optional[int] = None, layers: Optional[int] = None,
                  kernel_size: int = 3) -> Workload:
    """Workload ``name`` with its coordinates, bf16 features and per-layer
    weights ([K^3, C_in, C_out] for kernel size K; the coordinates and
    features do not depend on K)."""
    coords, shape, batch, rng = make_coords(name, seed)
    c_in, c_out, n_layers = _CHANNELS[name]
    if layers is not None:
        n_layers = layers
    feats = bf16_normal(rng, (coords.shape[0], c_in))
    weights = [make_weights(rng, c_in, c_out, kernel_size ** 3) for _ in range(n_layers)]
    return Workload(name=name, coords=torch.from_numpy(coords), spatial_shape=shape,
                    batch_size=batch, c_in=c_in, c_out=c_out, feats=feats,
                    weights=weights, seed=BASE_SEED + CONFIG_NAMES.index(name) + 1
                    if seed is None else seed)


def random_cloud(seed: int, n: int, shape=(12, 12, 12), batch_size: int = 1,
                 c_in: int = 16, c_out: int = 16, dense: bool = False) -> Workload:
    """Small uniform cloud for parity tests: ``n`` cells spread over ``batch_size`` frames."""
    rng = np.random.default_rng(seed)
    X, Y, Z = shape
    per = [n // batch_size + (1 if b < n % batch_size else 0) for b in range(batch_size)]
    parts = [uniform_cells(rng, per[b], shape, batch=b) for b in range(batch_size) if per[b]]
    coords = np.concatenate(parts, 0) if parts else np.zeros((0, 4), np.int32)
    coords = shuffle_rows(rng, coords)
    feats = bf16_normal(rng, (coords.shape[0], c_in))
    w = make_weights(rng, c_in, c_out)
    return Workload(name=f"random{n}", coords=torch.from_numpy(coords), spatial_shape=shape,
                    batch_size=batch_size, c_in=c_in, c_out=c_out, feats=feats,
                    weights=[w], seed=seed)
