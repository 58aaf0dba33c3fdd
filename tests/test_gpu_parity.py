"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Kernel maps, masks, row order and pair lists must match bit for bit.  bf16
outputs (fp32 accumulation, one rounding) must satisfy
|out - ref| <= 2e-2 * (1 + |ref|) against the fp64 oracle; fp32 exact-mode
outputs |out - ref| <= 1e-5.  Every case, the full-size workloads included,
compares every output row: the fp64 oracle evaluates all rows with its OpenMP
threads (each row summed by one thread in a fixed order).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import submanifold_sparse_convolution_gb300 as sc
from submanifold_sparse_convolution_gb300 import build as build_mod
from submanifold_sparse_convolution_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

BF16_RTOL = 2e-2
FP32_ATOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    oracle.build()


def oracle_map(coords, shape, batch, calibrated=True):
    nbr = oracle.kernel_map(coords, shape, batch)
    m = oracle.masks(nbr)
    p = oracle.perm(oracle.sort_keys(m, oracle.tap_order(m, calibrated)))
    tap_off, ins, outs = oracle.pair_lists(nbr, p)
    return dict(nbr=nbr, mask=m, perm=p, tap_off=tap_off, in_rows=ins, out_rows=outs)


def assert_map_equal(ex, ref):
    assert np.array_equal(ex["nbr"].cpu().numpy(), ref["nbr"])
    assert np.array_equal(ex["mask"].cpu().numpy().view(np.uint32), ref["mask"])
    assert np.array_equal(ex["perm"].cpu().numpy(), ref["perm"])
    assert np.array_equal(ex["tap_off"].cpu().numpy(), ref["tap_off"])
    assert np.array_equal(ex["in_rows"].cpu().numpy(), ref["in_rows"])
    assert np.array_equal(ex["out_rows"].cpu().numpy(), ref["out_rows"])


def check_bf16(out, ref):
    got = out.double().cpu().numpy()
    err = np.abs(got - ref)
    bound = BF16_RTOL * (1.0 + np.abs(ref))
    worst = float((err / bound).max()) if err.size else 0.0
    assert np.all(err <= bound), f"max err/bound {worst:.3f}"
    return worst


def check_fp32(out, ref):
    err = np.abs(out.double().cpu().numpy() - ref)
    assert err.size == 0 or err.max() <= FP32_ATOL, f"max abs err {err.max():.3e}"


def build(wl, mapper="auto", bit_order="calibrated", pipeline="auto", gemm="auto"):
    coords = wl.coords.cuda()
    m = sc.build_map(coords, wl.spatial_shape, wl.batch_size, mapper=mapper, bit_order=bit_order,
                     pipeline=pipeline, gemm=gemm)
    assert sc.map_status(m) == 0
    return m


# ---------------------------------------------------------------------------
# kernel map and pair lists
# ---------------------------------------------------------------------------

SMALL = [(1, 1, (4, 4, 4), 1), (2, 7, (5, 5, 5), 1), (3, 127, (8, 8, 8), 1), (4, 128, (8, 8, 8), 1),
         (5, 129, (8, 8, 8), 2), (6, 1000, (12, 12, 12), 3), (7, 5000, (24, 24, 24), 2),
         (8, 27, (3, 3, 3), 1), (9, 4096, (16, 16, 16), 1)]


@pytest.mark.parametrize("seed,n,shape,batch", SMALL)
@pytest.mark.parametrize("mapper", ["dense", "sorted"])
@pytest.mark.parametrize("bit_order", ["calibrated", "plain"])
@pytest.mark.parametrize("pipeline", ["fused", "multi", "wide"])
def test_map_small(seed, n, shape, batch, mapper, bit_order, pipeline):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch)
    m = build(wl, mapper, bit_order, pipeline)
    ref = oracle_map(wl.coords.numpy(), shape, batch, bit_order == "calibrated")
    assert_map_equal(sc.map_export(m), ref)
    info = sc.map_info(m)
    assert info["mapper"] == mapper and info["pairs"] == int(ref["tap_off"][27])
    assert info["pipeline"] == pipeline


@pytest.mark.parametrize("name", ["tiny", "outdoor", "deep", "large", "stage"])
@pytest.mark.parametrize("pipeline", ["auto", "fused", "multi"])
def test_map_workloads(name, pipeline):
    coords, shape, batch, _ = S.make_coords(name)
    wl = S.Workload(name, torch.from_numpy(coords), shape, batch, 1, 1, None, [], 0)
    m = build(wl, pipeline=pipeline)
    ref = oracle_map(coords, shape, batch)
    ex = sc.map_export(m)
    assert_map_equal(ex, ref)
    info = ex["info"]
    # AUTO: the dense grid on the small boxes; keys elsewhere, hashed by the whole-GPU pipeline
    assert info["mapper"] == ("dense" if name in ("tiny", "deep") else ("hash" if pipeline == "auto" else "sorted"))
    assert info["pipeline"] == ("wide" if pipeline == "auto" else pipeline)


@pytest.mark.parametrize("name", ["outdoor", "large", "stage"])
def test_map_workloads_wide_sorted(name):
    # the sorted mapper on the whole-GPU pipeline (AUTO hashes these workloads)
    coords, shape, batch, _ = S.make_coords(name)
    wl = S.Workload(name, torch.from_numpy(coords), shape, batch, 1, 1, None, [], 0)
    ex = sc.map_export(build(wl, "sorted", pipeline="wide"))
    assert_map_equal(ex, oracle_map(coords, shape, batch))
    assert ex["info"]["mapper"] == "sorted" and ex["info"]["pipeline"] == "wide"


@pytest.mark.parametrize("seed,n,shape,batch", SMALL)
@pytest.mark.parametrize("bit_order", ["calibrated", "plain"])
def test_map_small_hash(seed, n, shape, batch, bit_order):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch)
    m = build(wl, "hash", bit_order, "wide")
    ref = oracle_map(wl.coords.numpy(), shape, batch, bit_order == "calibrated")
    assert_map_equal(sc.map_export(m), ref)
    assert sc.map_info(m)["mapper"] == "hash"


def _hash_bucket_of_pairs(keys, lb):
    """The library's bucket of each key's z pair (multiplicative hashing of key >> 1), restated
    here to build a cloud that overfills buckets."""
    phi = np.uint64(0x9E3779B97F4A7C15)
    with np.errstate(over="ignore"):
        return ((keys >> np.uint64(1)) * phi) >> np.uint64(64 - lb)


def test_map_hash_full_buckets():
    """Pairs of voxels chosen so that many hash to one bucket: insertion overflows into the
    following buckets and lookups take the extra rounds; the map must still be exact."""
    shape, n_target = (64, 64, 64), 480
    X, Y, Z = shape
    wz, wy, wx = (Z + 1).bit_length(), (Y + 1).bit_length(), (X + 1).bit_length()
    log2 = 11
    while (1 << log2) < 16 * n_target:
        log2 += 1
    lb = log2 - 2
    g = np.stack(np.meshgrid(np.arange(X), np.arange(Y), np.arange(0, Z, 2), indexing="ij"), -1).reshape(-1, 3)
    g = g.astype(np.uint64)
    keys = (((g[:, 0] + 1) << np.uint64(wy) | (g[:, 1] + 1)) << np.uint64(wz)) | (g[:, 2] + 1)
    buckets = _hash_bucket_of_pairs(keys, lb)
    target = np.bincount(buckets.astype(np.int64)).argmax()
    hot = g[buckets == target][:16].astype(np.int64)          # 16 distinct pairs in one bucket
    assert hot.shape[0] == 16
    rng = np.random.default_rng(861)
    cells = {tuple(v) for v in hot}
    cells |= {(x, y, z + 1) for x, y, z in hot if z + 1 < Z}   # a voxel above each
    for x, y, z in hot:                                        # neighbours that look them up
        for d in rng.integers(-1, 2, size=(6, 3)):
            c = (x + d[0], y + d[1], z + d[2])
            if all(0 <= c[i] < shape[i] for i in range(3)):
                cells.add(tuple(int(v) for v in c))
    while len(cells) < n_target:
        cells.add(tuple(int(v) for v in rng.integers(0, 64, size=3)))
    coords = np.array([(0,) + c for c in sorted(cells)], dtype=np.int32)
    coords = coords[rng.permutation(len(coords))]
    assert 16 * len(coords) <= (1 << log2) and 16 * len(coords) > (1 << (log2 - 1))
    m = sc.build_map(torch.from_numpy(coords).cuda(), shape, 1, mapper="hash")
    assert sc.map_status(m) == 0
    assert_map_equal(sc.map_export(m), oracle_map(coords, shape, 1))


def test_map_hash_many_rows_and_unsupported_pipelines():
    """300k rows in 3 frames (a 2M-slot table): the hash and sorted mappers give the same map;
    the hash mapper exists only in the whole-GPU pipeline."""
    wl = S.random_cloud(63, 300000, shape=(200, 200, 60), batch_size=3)
    a = sc.map_export(build(wl, "hash", pipeline="wide"))
    b = sc.map_export(build(wl, "sorted", pipeline="wide"))
    for key in ("nbr", "mask", "perm", "tap_off", "in_rows", "out_rows"):
        assert torch.equal(a[key], b[key]), key
    for pipeline in ("fused", "multi"):
        with pytest.raises(sc.SpconvError) as e:
            sc.build_map(wl.coords.cuda(), wl.spatial_shape, 3, mapper="hash", pipeline=pipeline)
        assert e.value.code == -2



@pytest.mark.parametrize("mapper", ["sorted", "dense"])
def test_map_many_rows_pipelines_agree(mapper):
    """Several ranking rounds and tiles per CTA in the cluster pipeline, hundreds of
    look-back partitions in the whole-GPU one (N = 300k, 3 frames)."""
    wl = S.random_cloud(61, 300000, shape=(200, 200, 60), batch_size=3)
    b = sc.map_export(build(wl, mapper, pipeline="multi"))
    for pipeline in ("fused", "wide"):
        a = sc.map_export(build(wl, mapper, pipeline=pipeline))
        for key in ("nbr", "mask", "perm", "tap_off", "in_rows", "out_rows"):
            assert torch.equal(a[key], b[key]), (pipeline, key)


@pytest.mark.parametrize("y_extent", [1024, 2048])
@pytest.mark.parametrize("pipeline", ["wide", "fused"])
def test_map_sparse_line_beside_dense_slab(y_extent, pipeline):
    """A line of voxels at x = 10 next to a full (y, z) slab at x = 11: the sorted
    search's run for the slab column is y-range x 40 keys long, far beyond its
    shared-memory window, so it takes the in-place global search; 42k rows use
    the small-array block shape, 84k rows the large one."""
    rng = np.random.default_rng(71)
    line = np.stack([np.zeros(y_extent), np.full(y_extent, 10), np.arange(y_extent), np.zeros(y_extent)], 1)
    yy, zz = np.meshgrid(np.arange(y_extent), np.arange(40), indexing="ij")
    slab = np.stack([np.zeros(yy.size), np.full(yy.size, 11), yy.ravel(), zz.ravel()], 1)
    coords = np.concatenate([line, slab], 0).astype(np.int32)
    coords = coords[rng.permutation(len(coords))]
    shape = (16, y_extent, 40)
    m = sc.build_map(torch.from_numpy(coords).cuda(), shape, 1, mapper="sorted", pipeline=pipeline)
    assert sc.map_status(m) == 0
    assert_map_equal(sc.map_export(m), oracle_map(coords, shape, 1))


def test_map_ticketed_sort_passes_agree():
    """420k rows: more sort-pass CTAs (1024 keys each) than the GPU holds at once,
    so the whole-GPU passes take their partitions from ticket counters and use
    the look-back (not the grid barriers)."""
    wl = S.random_cloud(62, 420000, shape=(240, 240, 60), batch_size=2)
    a = sc.map_export(build(wl, "sorted", pipeline="wide"))
    b = sc.map_export(build(wl, "sorted", pipeline="multi"))
    for key in ("nbr", "mask", "perm", "tap_off", "in_rows", "out_rows"):
        assert torch.equal(a[key], b[key]), key


def test_map_recycled_arena():
    """Map memory is recycled between builds.  Look-back states of a sort pass left in it by
    earlier builds (or hash-table entries, whose top half can equal a pass's epoch) must not be
    taken for published ones: a 300k-row hash build, freed, then a 420k-row ticketed sorted build
    in the same memory, three times over, against the one-kernel-per-step pipeline."""
    big = S.random_cloud(64, 300000, shape=(200, 200, 60), batch_size=3)
    wl = S.random_cloud(62, 420000, shape=(240, 240, 60), batch_size=2)
    ref = sc.map_export(build(wl, "sorted", pipeline="multi"))
    for _ in range(3):
        build(big, "hash", pipeline="wide").destroy()
        a = sc.map_export(build(wl, "sorted", pipeline="wide"))
        for key in ("nbr", "mask", "perm", "tap_off", "in_rows", "out_rows"):
            assert torch.equal(a[key], ref[key]), key


@pytest.mark.parametrize("name", ["tiny", "deep"])
def test_dense_and_sorted_mappers_agree(name):
    coords, shape, batch, _ = S.make_coords(name)
    wl = S.Workload(name, torch.from_numpy(coords), shape, batch, 1, 1, None, [], 0)
    a = sc.map_export(build(wl, "dense"))
    for mapper in ("sorted", "hash"):
        b = sc.map_export(build(wl, mapper))
        for key in ("nbr", "mask", "perm", "tap_off", "in_rows", "out_rows"):
            assert torch.equal(a[key], b[key]), (mapper, key)


def test_dense_mapper_past_the_self_scanning_tile_limits():
    """A dense-grid map with more tiles than the tile writes that scan for
    themselves take (1024 for one group, 512 per group): the tile scans then
    start every tap's list from the per-tap totals the grid lookup counted.
    Kernel size 3 against the oracle and the hash mapper; kernel size 5 (five
    groups, 1,172 tiles each) against the sorted mapper."""
    wl = S.random_cloud(61, 150000, shape=(160, 160, 160))
    a = sc.map_export(build(wl, "dense", pipeline="wide"))
    assert a["info"]["mapper"] == "dense" and a["info"]["n_tiles"] > 1024
    assert_map_equal(a, oracle_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size))
    b = sc.map_export(build(wl, "hash", pipeline="wide"))
    for key in ("nbr", "mask", "perm", "tap_off", "in_rows", "out_rows"):
        assert torch.equal(a[key], b[key]), key
    c5 = wl.coords.cuda()
    d5 = sc.build_map(c5, wl.spatial_shape, 1, kernel_size=5, mapper="dense")
    s5 = sc.build_map(c5, wl.spatial_shape, 1, kernel_size=5, mapper="sorted")
    assert sc.map_status(d5) == 0 and sc.map_status(s5) == 0
    ed, es = sc.map_export(d5), sc.map_export(s5)
    assert ed["info"]["mapper"] == "dense" and ed["info"]["groups"] == 5
    for key in ("nbr", "mask", "perm", "tap_off", "in_rows", "out_rows"):
        assert torch.equal(ed[key], es[key]), key


def test_derived_shape_and_batch():
    wl = S.random_cloud(21, 900, shape=(10, 11, 12), batch_size=3)
    explicit = sc.map_export(build(wl))
    m = sc.build_map(wl.coords.cuda())          # shape and batch derived on the device
    info = sc.map_info(m)
    c = wl.coords.numpy()
    assert info["batch_size"] == int(c[:, 0].max()) + 1
    assert info["shape"] == tuple(int(v) + 1 for v in c[:, 1:].max(0))
    derived = sc.map_export(m)
    for key in ("nbr", "mask", "in_rows", "out_rows"):
        assert torch.equal(explicit[key], derived[key]), key


def test_empty_input():
    coords = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    m = sc.build_map(coords, (4, 4, 4), 1)
    assert sc.map_status(m) == 0
    assert sc.map_info(m)["pairs"] == 0
    out = sc.subm_forward(m, torch.zeros((0, 16), dtype=torch.bfloat16, device="cuda"),
                          torch.zeros((27, 16, 16), dtype=torch.bfloat16, device="cuda"))
    assert out.shape == (0, 16)


@pytest.mark.parametrize("pipeline", ["fused", "multi", "wide"])
def test_duplicate_and_range_errors(pipeline):
    dup = torch.tensor([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=torch.int32, device="cuda")
    mappers = ("dense", "sorted", "hash") if pipeline == "wide" else ("dense", "sorted")
    for mapper in mappers:
        m = sc.build_map(dup, (4, 4, 4), 1, mapper=mapper, pipeline=pipeline)
        assert sc.map_status(m) == -5
    bad = torch.tensor([[0, 1, 1, 1], [0, 4, 0, 0]], dtype=torch.int32, device="cuda")
    for mapper in mappers:
        m = sc.build_map(bad, (4, 4, 4), 1, mapper=mapper, pipeline=pipeline)
        assert sc.map_status(m) == -6
    neg = torch.tensor([[0, 1, 1, 1], [0, -1, 0, 0]], dtype=torch.int32, device="cuda")
    with pytest.raises(sc.SpconvError):
        sc.build_map(neg)                       # derived shape sees the negative coordinate


def test_alias_rejected():
    wl = S.random_cloud(22, 300, shape=(8, 8, 8), c_in=16, c_out=16)
    m = build(wl)
    buf = torch.zeros((300, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sc.SpconvError) as e:
        sc.subm_forward(m, buf, wl.weights[0].cuda(), out=buf)
    assert e.value.code == -7


# ---------------------------------------------------------------------------
# features
# ---------------------------------------------------------------------------

CHANNELS = [(16, 16), (64, 64), (128, 128), (24, 48), (8, 32), (256, 512), (512, 512), (3, 5), (1, 1),
            (16, 20)]


@pytest.mark.parametrize("c_in,c_out", CHANNELS)
def test_bf16_forward_small(c_in, c_out):
    wl = S.random_cloud(100 + c_in + c_out, 1500, shape=(14, 14, 14), batch_size=2, c_in=c_in, c_out=c_out)
    m = build(wl)
    out = sc.subm_forward(m, wl.feats.cuda(), wl.weights[0].cuda())
    assert sc.map_status(m) == 0
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    ref = oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy())
    check_bf16(out, ref)


@pytest.mark.parametrize("n", [1, 50, 1300, 4100])
def test_bf16_c128_tile_pairs(n):
    # ragged and single-tile inputs at C_out = 128 (one output block of the
    # tensor-core kernel): a lone voxel, a short tile, odd tile counts
    wl = S.random_cloud(400 + n, n, shape=(20, 20, 20), batch_size=1, c_in=128, c_out=128)
    m = build(wl)
    f, w = wl.feats.cuda(), wl.weights[0].cuda()
    out = sc.subm_forward(m, f, w)
    assert sc.map_status(m) == 0
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    check_bf16(out, oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy()))
    # a second call on the same map gives the same bits
    assert torch.equal(out, sc.subm_forward(m, f, w))


@pytest.mark.parametrize("c_in,c_out", CHANNELS)
def test_bf16_tap_major_small(c_in, c_out):
    # the tap-major decomposition: same sums, fp32 atomics, one rounding
    wl = S.random_cloud(300 + c_in + c_out, 1500, shape=(14, 14, 14), batch_size=2, c_in=c_in, c_out=c_out)
    m = build(wl, gemm="tap_major")
    assert sc.map_info(m)["gemm"] == "tap_major"
    out = sc.subm_forward(m, wl.feats.cuda(), wl.weights[0].cuda())
    assert sc.map_status(m) == 0
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    ref = oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy())
    check_bf16(out, ref)
    # a second call on the same map (the fp32 workspace is reused and cleared)
    check_bf16(sc.subm_forward(m, wl.feats.cuda(), wl.weights[0].cuda()), ref)


@pytest.mark.parametrize("c_in,c_out", [(64, 64), (16, 16), (5, 7), (128, 128)])
def test_fp32_exact_small(c_in, c_out):
    wl = S.random_cloud(200 + c_in, 2000, shape=(14, 14, 14), c_in=c_in, c_out=c_out)
    rng = np.random.default_rng(201)
    f = torch.from_numpy(rng.standard_normal((wl.n, c_in)).astype(np.float32))
    w = torch.from_numpy((rng.standard_normal((27, c_in, c_out)) * S.weights_std(c_in)).astype(np.float32))
    m = build(wl)
    out = sc.subm_forward(m, f.cuda(), w.cuda())
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    check_fp32(out, oracle.conv_f64(nbr, f.double().numpy(), w.double().numpy()))


@pytest.mark.parametrize("c_in,c_out,n", [(64, 64, 3000), (128, 128, 2000), (64, 192, 700), (100, 64, 1500)])
def test_fp32_tiled_matches_generic_bits(c_in, c_out, n):
    """The tiled fp32 kernel (16-byte aligned buffers) and the one-thread-per-output kernel
    (reached through a misaligned output view) run the same FMA chain: equal bits, with an
    epilogue, and within 1e-5 of the oracle."""
    wl = S.random_cloud(700 + c_in + n, n, shape=(16, 16, 16), batch_size=2, c_in=c_in, c_out=c_out)
    rng = np.random.default_rng(701)
    f = torch.from_numpy(rng.standard_normal((wl.n, c_in)).astype(np.float32)).cuda()
    w = torch.from_numpy((rng.standard_normal((27, c_in, c_out)) * S.weights_std(c_in)).astype(np.float32)).cuda()
    bias = torch.from_numpy(rng.standard_normal(c_out).astype(np.float32)).cuda()
    m = build(wl)
    a = sc.subm_forward(m, f, w, bias=bias, relu=True)
    big = torch.empty(wl.n * c_out + 1, dtype=torch.float32, device="cuda")
    b = sc.subm_forward(m, f, w, out=big[1:].view(wl.n, c_out), bias=bias, relu=True)
    assert sc.map_status(m) == 0
    assert torch.equal(a, b)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    ref = oracle.epilogue_f64(oracle.conv_f64(nbr, f.double().cpu().numpy(), w.double().cpu().numpy()),
                              bias=bias.double().cpu().numpy(), relu=True)
    check_fp32(a, ref)


def test_packed_weights_match_unpacked():
    wl = S.random_cloud(31, 3000, shape=(16, 16, 16), c_in=128, c_out=128)
    m = build(wl)
    f, w = wl.feats.cuda(), wl.weights[0].cuda()
    a = sc.subm_forward(m, f, w)
    wp = sc.wpack_create(w)
    b = sc.subm_forward_packed(m, f, wp)
    c = sc.subm_forward_packed(m, f, wp)
    assert torch.equal(a, b) and torch.equal(b, c)


def test_row_permutation_equivariance():
    wl = S.random_cloud(41, 2500, shape=(16, 16, 16), c_in=64, c_out=64)
    q = torch.from_numpy(np.random.default_rng(42).permutation(wl.n))
    m1, m2 = build(wl), None
    out1 = sc.subm_forward(m1, wl.feats.cuda(), wl.weights[0].cuda())
    coords2 = wl.coords[q].contiguous().cuda()
    m2 = sc.build_map(coords2, wl.spatial_shape, 1)
    out2 = sc.subm_forward(m2, wl.feats[q].contiguous().cuda(), wl.weights[0].cuda())
    torch.testing.assert_close(out2.float(), out1[q.cuda()].float(), rtol=1e-2, atol=1e-2)


def test_isolated_voxels_use_centre_tap_only():
    coords = torch.tensor([[0, 0, 0, 0], [0, 5, 5, 5], [0, 9, 2, 7], [1, 3, 3, 3]], dtype=torch.int32)
    rng = np.random.default_rng(43)
    f = torch.from_numpy(rng.standard_normal((4, 128)).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy((rng.standard_normal((27, 128, 128)) * 0.05).astype(np.float32)).to(torch.bfloat16)
    m = sc.build_map(coords.cuda(), (10, 10, 10), 2)
    out = sc.subm_forward(m, f.cuda(), w.cuda())
    ref = f.double().numpy() @ w[13].double().numpy()
    check_bf16(out, ref)


@pytest.mark.parametrize("name", ["tiny", "outdoor", "deep", "large"])
def test_bf16_workloads(name):
    wl = S.make_workload(name)
    m = build(wl)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    f, w = wl.feats.cuda(), wl.weights[0].cuda()
    wp = sc.wpack_create(w)
    out = sc.subm_forward_packed(m, f, wp)
    assert sc.map_status(m) == 0
    ref = oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy())
    check_bf16(out, ref)
    # the unpacked entry point gives the same bits
    assert torch.equal(out, sc.subm_forward(m, f, w))


@pytest.mark.parametrize("name", ["outdoor", "deep", "large"])
def test_bf16_workloads_tap_major(name):
    wl = S.make_workload(name)
    m = build(wl, gemm="tap_major")
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    out = sc.subm_forward_packed(m, wl.feats.cuda(), sc.wpack_create(wl.weights[0].cuda()))
    assert sc.map_status(m) == 0
    ref = oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy())
    check_bf16(out, ref)


def test_stage_six_layers_and_fp32_layer():
    wl = S.make_workload("stage")
    m = build(wl)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    x = wl.feats.cuda()
    for layer, w in enumerate(wl.weights):
        relu = layer + 1 < len(wl.weights)   # the ReLU between layers, fused into the store
        y = sc.subm_forward(m, x, w.cuda(), relu=relu)
        ref = oracle.epilogue_f64(oracle.conv_f64(nbr, x.double().cpu().numpy(), w.double().numpy()), relu=relu)
        check_bf16(y, ref)
        x = y
    # the first layer again in exact fp32
    f32 = wl.feats.float().cuda()
    w32 = wl.weights[0].float().cuda()
    y32 = sc.subm_forward(m, f32, w32)
    ref = oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy())
    check_fp32(y32, ref)


# ---------------------------------------------------------------------------
# fused epilogue (scale, bias, residual, ReLU)
# ---------------------------------------------------------------------------

EPI_CASES = [  # (c_in, c_out, dtype, gemm): tensor-core tile-union and tap-major, SIMT bf16, fp32
    (64, 64, torch.bfloat16, "tile_union"), (128, 128, torch.bfloat16, "tile_union"),
    (32, 256, torch.bfloat16, "tile_union"), (128, 128, torch.bfloat16, "tap_major"),
    (5, 7, torch.bfloat16, "tile_union"), (16, 16, torch.float32, "tile_union")]
EPI_TERMS = [dict(relu=True), dict(bias=True), dict(scale=True, bias=True),
             dict(residual=True), dict(scale=True, bias=True, residual=True, relu=True)]


def epilogue_inputs(n, c_out, dtype, terms, seed):
    rng = np.random.default_rng(seed)
    scale = torch.from_numpy(rng.uniform(0.5, 1.5, c_out).astype(np.float32)) if terms.get("scale") else None
    bias = torch.from_numpy((rng.standard_normal(c_out) * 0.5).astype(np.float32)) if terms.get("bias") else None
    res = (torch.from_numpy(rng.standard_normal((n, c_out)).astype(np.float32)).to(dtype)
           if terms.get("residual") else None)
    return scale, bias, res


@pytest.mark.parametrize("c_in,c_out,dtype,gemm", EPI_CASES)
@pytest.mark.parametrize("ti", range(len(EPI_TERMS)))
def test_epilogue_forward(c_in, c_out, dtype, gemm, ti):
    terms = EPI_TERMS[ti]
    wl = S.random_cloud(600 + c_in + ti, 1700, shape=(14, 14, 14), batch_size=2, c_in=c_in, c_out=c_out)
    f, w = wl.feats.to(dtype), wl.weights[0].to(dtype)
    scale, bias, res = epilogue_inputs(wl.n, c_out, dtype, terms, 601 + ti)
    m = build(wl, gemm=gemm)
    cu = lambda t: None if t is None else t.cuda()
    out = sc.subm_forward(m, f.cuda(), w.cuda(), scale=cu(scale), bias=cu(bias), residual=cu(res),
                          relu=terms.get("relu", False))
    assert sc.map_status(m) == 0
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    conv = oracle.conv_f64(nbr, f.double().numpy(), w.double().numpy())
    d = lambda t: None if t is None else t.double().numpy()
    ref = oracle.epilogue_f64(conv, d(scale), d(bias), d(res), terms.get("relu", False))
    (check_fp32 if dtype == torch.float32 else check_bf16)(out, ref)
    # the packed-weight entry point applies the same epilogue to the same bits
    wp = sc.wpack_create(w.cuda())
    out2 = sc.subm_forward_packed(m, f.cuda(), wp, scale=cu(scale), bias=cu(bias), residual=cu(res),
                                  relu=terms.get("relu", False))
    if gemm == "tap_major":
        (check_fp32 if dtype == torch.float32 else check_bf16)(out2, ref)
    else:
        assert torch.equal(out, out2)


@pytest.mark.parametrize("gemm", ["tile_union", "tap_major"])
def test_epilogue_relu_equals_relu_of_output(gemm):
    # max(., 0) commutes with the rounding to bf16, so the fused ReLU gives
    # exactly the bits of a ReLU applied to the plain output
    wl = S.random_cloud(611, 5000, shape=(24, 24, 24), c_in=64, c_out=64)
    m = build(wl, gemm=gemm)
    f, w = wl.feats.cuda(), wl.weights[0].cuda()
    wp = sc.wpack_create(w)
    plain = sc.subm_forward_packed(m, f, wp)
    fused = sc.subm_forward_packed(m, f, wp, relu=True)
    if gemm == "tile_union":
        assert torch.equal(fused, torch.relu(plain))
    else:
        # tap-major sums in a run-dependent order; compare with the tolerance
        ref = oracle.epilogue_f64(oracle.conv_f64(oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1),
                                                  wl.feats.double().numpy(), wl.weights[0].double().numpy()),
                                  relu=True)
        check_bf16(fused, ref)
    assert (fused == 0).any() and (fused > 0).any()


def test_epilogue_residual_in_place():
    # residual == out: each element is read, then overwritten by the same thread
    wl = S.random_cloud(621, 3000, shape=(16, 16, 16), c_in=128, c_out=128)
    m = build(wl)
    rng = np.random.default_rng(622)
    r = torch.from_numpy(rng.standard_normal((wl.n, 128)).astype(np.float32)).to(torch.bfloat16)
    buf = r.cuda().clone()
    out = sc.subm_forward(m, wl.feats.cuda(), wl.weights[0].cuda(), out=buf, residual=buf, relu=True)
    assert out.data_ptr() == buf.data_ptr()
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    ref = oracle.epilogue_f64(oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy()),
                              residual=r.double().numpy(), relu=True)
    check_bf16(out, ref)


def test_epilogue_argument_errors():
    wl = S.random_cloud(631, 500, shape=(10, 10, 10), c_in=16, c_out=16)
    m = build(wl)
    f, w = wl.feats.cuda(), wl.weights[0].cuda()
    lib = sc.library()
    out = torch.empty((wl.n, 16), dtype=torch.bfloat16, device="cuda")
    import ctypes
    from submanifold_sparse_convolution_gb300 import _native

    def call(e):
        return lib.spconv_subm_forward_ex(m.handle, f.data_ptr(), w.data_ptr(), out.data_ptr(), 16, 16, 0,
                                          ctypes.byref(e), None)

    bias = torch.zeros(17, dtype=torch.float32, device="cuda")
    assert call(_native.Epilogue(None, None, None, 2)) == -1            # relu must be 0 or 1
    assert call(_native.Epilogue(None, bias.data_ptr() + 4, None, 0)) == -1   # bias not 16-byte aligned
    big = torch.empty((wl.n + 8, 16), dtype=torch.bfloat16, device="cuda")
    out = big[:wl.n]
    assert call(_native.Epilogue(None, None, big[8:].data_ptr(), 0)) == -7  # residual partly overlaps out
    assert call(_native.Epilogue(None, None, out.data_ptr(), 0)) == 0       # in place is allowed
    assert lib.spconv_subm_forward_ex(m.handle, f.data_ptr(), w.data_ptr(), out.data_ptr(), 16, 16, 0,
                                      None, None) == 0                     # NULL: the plain forward
    assert sc.map_status(m) == 0


@pytest.mark.parametrize("gemm", ["tile_union", "tap_major"])
def test_epilogue_full_outdoor(gemm):
    """Scale, bias, residual and ReLU together on the outdoor workload (32,371 rows, C = 128),
    every row against the oracle's convolution and epilogue."""
    wl = S.make_workload("outdoor")
    terms = dict(scale=True, bias=True, residual=True, relu=True)
    scale, bias, res = epilogue_inputs(wl.n, wl.c_out, torch.bfloat16, terms, 641)
    m = build(wl, gemm=gemm)
    out = sc.subm_forward_packed(m, wl.feats.cuda(), sc.wpack_create(wl.weights[0].cuda()), scale=scale.cuda(),
                                 bias=bias.cuda(), residual=res.cuda(), relu=True)
    assert sc.map_status(m) == 0
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    conv = oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy())
    check_bf16(out, oracle.epilogue_f64(conv, scale.double().numpy(), bias.double().numpy(),
                                        res.double().numpy(), relu=True))


# ---------------------------------------------------------------------------
# kernel size 5 and offset groups
# ---------------------------------------------------------------------------

def oracle_groups(coords, shape, batch, K, G, calibrated=True):
    nbr = oracle.kernel_map(coords, shape, batch, K)
    m, _, p = oracle.group_orders(nbr, G, calibrated)
    tap_off, ins, outs = oracle.pair_lists(nbr, p)
    if G == 1:
        m, p = m[0], p[0]
    return dict(nbr=nbr, mask=m, perm=p, tap_off=tap_off, in_rows=ins, out_rows=outs)


def weights_k(K, c_in, c_out, seed, dtype=torch.bfloat16):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((K ** 3, c_in, c_out)) / np.sqrt(K ** 3 * c_in)
    return torch.from_numpy(w.astype(np.float32)).to(dtype)


GROUP_CASES = [(3, 3), (5, 5)]
GROUP_SMALL = [(1, 1, (4, 4, 4), 1), (2, 7, (5, 5, 5), 1), (3, 128, (8, 8, 8), 1), (4, 129, (8, 8, 8), 2),
               (5, 1500, (14, 13, 12), 2), (6, 4000, (30, 30, 6), 1)]


@pytest.mark.parametrize("K,G", GROUP_CASES)
@pytest.mark.parametrize("seed,n,shape,batch", GROUP_SMALL)
@pytest.mark.parametrize("mapper", ["dense", "sorted", "hash"])
@pytest.mark.parametrize("bit_order", ["calibrated", "plain"])
def test_map_groups_small(K, G, seed, n, shape, batch, mapper, bit_order):
    wl = S.random_cloud(700 + seed, n, shape=shape, batch_size=batch)
    m = sc.build_map(wl.coords.cuda(), shape, batch, kernel_size=K, groups=G, mapper=mapper, bit_order=bit_order)
    assert sc.map_status(m) == 0
    info = sc.map_info(m)
    assert info["kernel_size"] == K and info["groups"] == G and info["mapper"] == mapper
    ex = sc.map_export(m)
    ref = oracle_groups(wl.coords.numpy(), shape, batch, K, G, bit_order == "calibrated")
    assert_map_equal(ex, ref)
    assert info["pairs"] == ref["tap_off"][-1]


@pytest.mark.parametrize("K,G", GROUP_CASES)
def test_map_groups_dense_and_sorted_agree_on_outdoor(K, G):
    wl = S.make_workload("outdoor")
    ref = oracle_groups(wl.coords.numpy(), wl.spatial_shape, wl.batch_size, K, G)
    for mapper in ("sorted", "dense", "hash"):
        m = sc.build_map(wl.coords.cuda(), wl.spatial_shape, wl.batch_size, kernel_size=K, groups=G,
                         mapper=mapper, dense_max_cells=1 << 30)
        assert sc.map_status(m) == 0
        assert_map_equal(sc.map_export(m), ref)


FWD_GROUP = [(64, 64, torch.bfloat16), (128, 128, torch.bfloat16), (32, 256, torch.bfloat16),
             (16, 16, torch.bfloat16), (5, 7, torch.bfloat16), (16, 16, torch.float32)]


@pytest.mark.parametrize("K,G", GROUP_CASES)
@pytest.mark.parametrize("c_in,c_out,dtype", FWD_GROUP)
def test_forward_groups(K, G, c_in, c_out, dtype):
    wl = S.random_cloud(800 + c_in + K, 2500, shape=(16, 16, 16), batch_size=2, c_in=c_in, c_out=c_out)
    f = wl.feats.to(dtype)
    w = weights_k(K, c_in, c_out, 801 + c_out, dtype)
    m = sc.build_map(wl.coords.cuda(), wl.spatial_shape, wl.batch_size, kernel_size=K, groups=G)
    out = sc.subm_forward(m, f.cuda(), w.cuda())
    assert sc.map_status(m) == 0
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size, K)
    ref = oracle.conv_f64(nbr, f.double().numpy(), w.double().numpy())
    (check_fp32 if dtype == torch.float32 else check_bf16)(out, ref)
    # packed weights: the same bits; a pack for another kernel size is refused
    wp = sc.wpack_create(w.cuda())
    assert torch.equal(sc.subm_forward_packed(m, f.cuda(), wp), out)
    other = sc.wpack_create(weights_k(8 - K, c_in, c_out, 5, dtype).cuda())
    with pytest.raises(ValueError):
        sc.subm_forward_packed(m, f.cuda(), other)
    rc = sc.library().spconv_subm_forward_packed(m.handle, f.cuda().data_ptr(), other.handle,
                                                 out.data_ptr(), None)
    assert rc == -1


@pytest.mark.parametrize("K,G", GROUP_CASES)
def test_forward_groups_epilogue(K, G):
    # the epilogue is applied once, by the last group's pass, to every row
    wl = S.random_cloud(811 + K, 3000, shape=(18, 18, 18), c_in=64, c_out=64)
    w = weights_k(K, 64, 64, 812)
    scale, bias, res = epilogue_inputs(wl.n, 64, torch.bfloat16, dict(scale=1, bias=1, residual=1), 813)
    m = sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, kernel_size=K, groups=G)
    out = sc.subm_forward(m, wl.feats.cuda(), w.cuda(), scale=scale.cuda(), bias=bias.cuda(),
                          residual=res.cuda(), relu=True)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1, K)
    ref = oracle.epilogue_f64(oracle.conv_f64(nbr, wl.feats.double().numpy(), w.double().numpy()),
                              scale.double().numpy(), bias.double().numpy(), res.double().numpy(), True)
    check_bf16(out, ref)


def test_three_groups_match_one_group():
    # K = 3 in one group or in three: the same sums up to fp32 rounding order
    wl = S.random_cloud(821, 6000, shape=(24, 24, 24), c_in=128, c_out=128)
    f, w = wl.feats.cuda(), wl.weights[0].cuda()
    m1 = sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1)
    m3 = sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, groups=3)
    a, b = sc.subm_forward(m1, f, w), sc.subm_forward(m3, f, w)
    torch.testing.assert_close(a.float(), b.float(), rtol=2e-2, atol=2e-2)
    i1, i3 = sc.map_info(m1), sc.map_info(m3)
    assert i1["pairs"] == i3["pairs"]
    # each group's tiles cover only its own taps: fewer executed tile-taps than 3 x one group
    assert i3["tile_taps"] < 3 * i1["tile_taps"]


@pytest.mark.parametrize("name", ["outdoor", "stage"])
def test_k5_workload(name):
    wl = S.make_workload(name)
    K = 5
    w = weights_k(K, wl.c_in, wl.c_out, 831)
    m = sc.build_map(wl.coords.cuda(), wl.spatial_shape, wl.batch_size, kernel_size=K)
    out = sc.subm_forward(m, wl.feats.cuda(), w.cuda())
    assert sc.map_status(m) == 0
    ex = sc.map_export(m)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size, K)
    assert np.array_equal(ex["nbr"].cpu().numpy(), nbr)
    ref = oracle_groups(wl.coords.numpy(), wl.spatial_shape, wl.batch_size, K, K)
    assert_map_equal(ex, ref)
    check_bf16(out, oracle.conv_f64(nbr, wl.feats.double().numpy(), w.double().numpy()))


@pytest.mark.parametrize("K,G", GROUP_CASES)
def test_groups_with_empty_tiles(K, G):
    # voxels on even x only: no row has a dx = +-1 neighbour, so those groups
    # have no tile to visit at all, and a sparse tail gives runs of empty tiles
    rng = np.random.default_rng(851)
    lattice = np.array([(0, x, y, z) for x in range(0, 24, 2) for y in range(10) for z in range(10)], np.int32)
    tail = np.array([(0, 40 + 6 * i, 3 * (i % 3), 5) for i in range(300)], np.int32)
    coords = np.concatenate([lattice, tail])[rng.permutation(lattice.shape[0] + 300)]
    shape = (40 + 6 * 300, 10, 10)
    f = torch.from_numpy(rng.standard_normal((coords.shape[0], 64)).astype(np.float32)).to(torch.bfloat16)
    w = weights_k(K, 64, 64, 852)
    m = sc.build_map(torch.from_numpy(coords).cuda(), shape, 1, kernel_size=K, groups=G)
    out = sc.subm_forward(m, f.cuda(), w.cuda(), relu=True)
    assert sc.map_status(m) == 0
    ref_map = oracle_groups(coords, shape, 1, K, G)
    assert_map_equal(sc.map_export(m), ref_map)
    nbr = ref_map["nbr"]
    assert (nbr[:, K * K * ((K - 1) // 2 - 1):K * K * ((K - 1) // 2)] < 0).all()   # the dx = -1 group is empty
    check_bf16(out, oracle.epilogue_f64(oracle.conv_f64(nbr, f.double().numpy(), w.double().numpy()), relu=True))


def test_groups_argument_errors():
    wl = S.random_cloud(841, 300, shape=(8, 8, 8))
    c = wl.coords.cuda()
    for kw in (dict(kernel_size=5, groups=1), dict(kernel_size=3, groups=2), dict(kernel_size=7),
               dict(kernel_size=5, pipeline="wide"), dict(kernel_size=5, pipeline="fused"),
               dict(kernel_size=3, groups=3, gemm="tap_major"), dict(kernel_size=5, gemm="tap_major")):
        with pytest.raises(sc.SpconvError) as e:
            sc.build_map(c, wl.spatial_shape, 1, **kw)
        assert e.value.code == -2, kw
    with pytest.raises(sc.SpconvError) as e:
        sc.build_map(c, wl.spatial_shape, 1, groups=-1)
    assert e.value.code == -1


def test_groups_duplicate_and_range_errors():
    for mapper in ("dense", "sorted", "hash"):
        dup = torch.tensor([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=torch.int32).cuda()
        m = sc.build_map(dup, (8, 8, 8), 1, kernel_size=5, mapper=mapper)
        assert sc.map_status(m) == -5
        bad = torch.tensor([[0, 1, 1, 1], [0, 8, 2, 2]], dtype=torch.int32).cuda()
        m = sc.build_map(bad, (8, 8, 8), 1, kernel_size=5, mapper=mapper)
        assert sc.map_status(m) == -6


def test_groups_empty_input():
    c = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    m = sc.build_map(c, (4, 4, 4), 1, kernel_size=5)
    assert sc.map_status(m) == 0 and sc.map_info(m)["pairs"] == 0
    out = sc.subm_forward(m, torch.empty((0, 16), dtype=torch.bfloat16, device="cuda"),
                          weights_k(5, 16, 16, 1).cuda())
    assert out.shape == (0, 16)


# ---------------------------------------------------------------------------
# strided convolution (kernel 3, stride 2, padding 1) and its inverse
# ---------------------------------------------------------------------------

def oracle_strided(coords, shape, batch, calibrated=True):
    oc, nbr = oracle.strided_map(coords, shape, batch)
    m = oracle.masks(nbr)
    p = oracle.perm(oracle.sort_keys(m, oracle.tap_order(m, calibrated)))
    tap_off, ins, outs = oracle.pair_lists(nbr, p)
    return oc, dict(nbr=nbr, mask=m, perm=p, tap_off=tap_off, in_rows=ins, out_rows=outs)


def oracle_inverse(nbr_s, n_in, calibrated=True):
    inv = oracle.inverse_map(nbr_s, n_in)
    m = oracle.masks(inv)
    p = oracle.perm(oracle.sort_keys(m, oracle.tap_order(m, calibrated)))
    tap_off, ins, outs = oracle.pair_lists(inv, p)
    return dict(nbr=inv, mask=m, perm=p, tap_off=tap_off, in_rows=ins, out_rows=outs)


STRIDED_SMALL = [(1, 1, (4, 4, 4), 1), (2, 7, (5, 5, 5), 1), (3, 129, (8, 9, 10), 2), (4, 1500, (14, 13, 12), 2),
                 (5, 3000, (31, 30, 7), 1)]


@pytest.mark.parametrize("seed,n,shape,batch", STRIDED_SMALL)
@pytest.mark.parametrize("bit_order", ["calibrated", "plain"])
def test_strided_and_inverse_maps_small(seed, n, shape, batch, bit_order):
    wl = S.random_cloud(900 + seed, n, shape=shape, batch_size=batch)
    m = sc.build_map_strided(wl.coords.cuda(), shape, batch, bit_order=bit_order)
    assert sc.map_status(m) == 0
    oc, ref = oracle_strided(wl.coords.numpy(), shape, batch, bit_order == "calibrated")
    info = sc.map_info(m)
    assert info["conv"] == "strided" and info["n"] == oc.shape[0] and info["n_in"] == n
    assert info["out_shape"] == oracle.strided_shape(shape)
    assert np.array_equal(sc.map_out_coords(m).cpu().numpy(), oc)
    assert_map_equal(sc.map_export(m), ref)
    mi = sc.build_map_inverse(m, bit_order=bit_order)
    assert sc.map_status(mi) == 0
    assert sc.map_info(mi)["conv"] == "inverse" and sc.map_info(mi)["n_in"] == oc.shape[0]
    assert_map_equal(sc.map_export(mi), oracle_inverse(ref["nbr"], n, bit_order == "calibrated"))


STRIDED_FWD = [(64, 64, torch.bfloat16), (128, 128, torch.bfloat16), (32, 256, torch.bfloat16),
               (5, 7, torch.bfloat16), (16, 16, torch.float32), (64, 128, torch.float32)]


@pytest.mark.parametrize("c_in,c_out,dtype", STRIDED_FWD)
def test_strided_and_inverse_forward(c_in, c_out, dtype):
    wl = S.random_cloud(950 + c_in, 2500, shape=(16, 17, 15), batch_size=2, c_in=c_in, c_out=c_out)
    f = wl.feats.to(dtype)
    w = wl.weights[0].to(dtype)
    m = sc.build_map_strided(wl.coords.cuda(), wl.spatial_shape, 2)
    y = sc.subm_forward(m, f.cuda(), w.cuda())
    assert sc.map_status(m) == 0 and y.shape == (m.n, c_out)
    oc, nbr = oracle.strided_map(wl.coords.numpy(), wl.spatial_shape, 2)
    rows, rows_in = ctypes.c_int64(-1), ctypes.c_int64(-1)   # the host-side counts, no synchronisation
    assert sc.library().spconv_map_rows(m.handle, ctypes.byref(rows), ctypes.byref(rows_in)) == 0
    assert rows.value == m.n == oc.shape[0] and rows_in.value == wl.n == sc.map_info(m)["n_in"]
    check = check_fp32 if dtype == torch.float32 else check_bf16
    check(y, oracle.conv_f64(nbr, f.double().numpy(), w.double().numpy()))
    # the inverse convolution back onto the input sites, with its own weights and a fused ReLU
    rng = np.random.default_rng(951)
    w2 = torch.from_numpy((rng.standard_normal((27, c_out, c_in)) / np.sqrt(27 * c_out)).astype(np.float32)).to(dtype)
    mi = sc.build_map_inverse(m)
    z = sc.subm_forward(mi, y, w2.cuda(), relu=True)
    assert z.shape == (wl.n, c_in)
    inv = oracle.inverse_map(nbr, wl.n)
    check(z, oracle.epilogue_f64(oracle.conv_f64(inv, y.double().cpu().numpy(), w2.double().numpy()), relu=True))


@pytest.mark.parametrize("name", ["outdoor", "stage"])
def test_strided_workload(name):
    wl = S.make_workload(name)
    m = sc.build_map_strided(wl.coords.cuda(), wl.spatial_shape, wl.batch_size)
    y = sc.subm_forward(m, wl.feats.cuda(), wl.weights[0].cuda())
    assert sc.map_status(m) == 0
    oc, ref = oracle_strided(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    assert np.array_equal(sc.map_out_coords(m).cpu().numpy(), oc)
    assert_map_equal(sc.map_export(m), ref)
    check_bf16(y, oracle.conv_f64(ref["nbr"], wl.feats.double().numpy(), wl.weights[0].double().numpy()))
    if name == "outdoor":
        # the inverse convolution back onto the input sites, every row, with its own weights and a ReLU
        rng = np.random.default_rng(962)
        w2 = torch.from_numpy((rng.standard_normal((27, wl.c_out, wl.c_in)) * S.weights_std(wl.c_out))
                              .astype(np.float32)).to(torch.bfloat16)
        mi = sc.build_map_inverse(m)
        z = sc.subm_forward(mi, y, w2.cuda(), relu=True)
        assert sc.map_status(mi) == 0 and z.shape == (wl.n, wl.c_in)
        assert_map_equal(sc.map_export(mi), oracle_inverse(ref["nbr"], wl.n))
        inv = oracle.inverse_map(ref["nbr"], wl.n)
        check_bf16(z, oracle.epilogue_f64(oracle.conv_f64(inv, y.double().cpu().numpy(), w2.double().numpy()),
                                          relu=True))


def test_strided_errors():
    c = torch.tensor([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=torch.int32).cuda()
    m = sc.build_map_strided(c, (8, 8, 8), 1)
    assert sc.map_status(m) == -5                     # duplicates, found at insertion
    bad = torch.tensor([[0, 1, 1, 1], [0, 8, 2, 2]], dtype=torch.int32).cuda()
    assert sc.map_status(sc.build_map_strided(bad, (8, 8, 8), 1)) == -6
    for kw in (dict(kernel_size=5), dict(stride=1)):
        with pytest.raises(sc.SpconvError) as e:
            sc.build_map_strided(c[:2].contiguous(), (8, 8, 8), 1, **kw)
        assert e.value.code == -2
    sub = sc.build_map(c[:2].contiguous(), (8, 8, 8), 1)
    with pytest.raises(sc.SpconvError) as e:
        sc.build_map_inverse(sub)                     # only a strided map has an inverse
    assert e.value.code == -1
    with pytest.raises(sc.SpconvError):
        sc.map_out_coords(sub)
    empty = sc.build_map_strided(torch.empty((0, 4), dtype=torch.int32, device="cuda"), (4, 4, 4), 1)
    assert sc.map_status(empty) == 0 and empty.n == 0


def test_launch_count_reported():
    wl = S.random_cloud(51, 3000, shape=(16, 16, 16), c_in=64, c_out=64)
    m = sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, mapper="dense", pipeline="fused")
    assert sc.last_launch_count() == 2                # cluster build + whole-GPU compaction write
    sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, mapper="sorted", pipeline="fused")
    assert sc.last_launch_count() == 4                # cluster sort, search, cluster rest, write
    # (up to 1024 tiles the tile write also does the tile scan's work: no scan launch)
    # (up to 64 sort partitions the first mask pass makes the mask keys itself)
    sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, mapper="dense", pipeline="wide")
    assert sc.last_launch_count() == 8                # clear, scatter, lookup, 3 passes, tile count/write
    sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, mapper="sorted", pipeline="wide")
    assert sc.last_launch_count() == 10               # clear, keys, 2 passes (15-bit keys), search,
                                                      # 3 passes, tile count/write
    sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, mapper="hash", pipeline="wide")
    assert sc.last_launch_count() == 8                # clear, insert, lookup, 3 passes, tile count/write
    big = S.random_cloud(52, 140000, shape=(100, 100, 40))
    sc.build_map(big.coords.cuda(), big.spatial_shape, 1, mapper="hash", pipeline="wide")
    assert sc.last_launch_count() == 9                # 35 partitions of 4096 keys; 1094 tiles: tile count,
                                                      # the tile scan, tile write
    bigger = S.random_cloud(53, 300000, shape=(100, 100, 40))
    sc.build_map(bigger.coords.cuda(), bigger.spatial_shape, 1, mapper="hash", pipeline="wide")
    assert sc.last_launch_count() == 10               # 74 partitions: the mask-key kernel; the tile scan
    sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, pipeline="multi")
    assert sc.last_launch_count() > 5
    # kernel size 5 (5 groups), sorted keys; every whole-GPU pass counted once
    sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, kernel_size=5, mapper="sorted")
    assert sc.last_launch_count() == 10         # pack, 2 passes (16-bit keys), search, mask keys,
                                                # 3 passes, tile count/write
    sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, groups=3, mapper="hash")
    assert sc.last_launch_count() == 7          # insert, lookup, mask keys, 2 passes (11-bit keys),
                                                # tile count/write
    sc.subm_forward(m, wl.feats.cuda(), wl.weights[0].cuda())
    assert sc.last_launch_count() == 2          # weight pack + GEMM
    mt = sc.build_map(wl.coords.cuda(), wl.spatial_shape, 1, gemm="tap_major")
    sc.subm_forward(mt, wl.feats.cuda(), wl.weights[0].cuda())
    assert sc.last_launch_count() == 3          # weight pack + GEMM + bf16 rounding pass


@pytest.mark.parametrize("which", [0, 1, 2])
def test_bounded_wait_times_out_and_gpu_keeps_working(which):
    """A sort pass's look-back (0), grid barrier (1) or predecessor flag (2) waits on a state
    that nothing publishes, with a 50 ms limit: it gives up, the call reports
    SPCONV_ERR_TIMEOUT, and the context still builds and convolves correctly afterwards."""
    import time
    lib = sc.library()
    stream = torch.cuda.current_stream().cuda_stream
    t = time.perf_counter()
    assert lib.spconv_selftest_wait_timeout(which, 50_000_000, stream) == -8
    assert time.perf_counter() - t < 10.0
    assert lib.spconv_selftest_wait_timeout(3, 50_000_000, stream) == -1
    assert lib.spconv_selftest_wait_timeout(which, 10, stream) == -1
    wl = S.random_cloud(881, 3000, shape=(16, 16, 16), c_in=64, c_out=64)
    m = build(wl)
    out = sc.subm_forward(m, wl.feats.cuda(), wl.weights[0].cuda())
    assert sc.map_status(m) == 0
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    check_bf16(out, oracle.conv_f64(nbr, wl.feats.double().numpy(), wl.weights[0].double().numpy()))


# ---------------------------------------------------------------------------
# a stack of layers over one map in one launch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("c,n,layers", [(64, 3000, 3), (128, 5000, 2), (64, 300, 4), (16, 1000, 2)])
def test_fused_layers_match_separate_layers(c, n, layers):
    """Every layer of the fused launch has the bits of the same layer run as its own launch
    (fewer items than SMs for n = 300: a smaller cooperative grid)."""
    wl = S.random_cloud(900 + c + n, n, shape=(20, 20, 20), batch_size=2, c_in=c, c_out=c)
    m = build(wl)
    rng = np.random.default_rng(901)
    ws = [torch.from_numpy((rng.standard_normal((27, c, c)) * S.weights_std(c)).astype(np.float32))
          .to(torch.bfloat16).cuda() for _ in range(layers)]
    wps = [sc.wpack_create(w) for w in ws]
    relu = [l + 1 < layers for l in range(layers)]
    outs = [torch.empty((wl.n, c), dtype=torch.bfloat16, device="cuda") for _ in range(layers)]
    fused = sc.subm_forward_layers(m, wl.feats.cuda(), wps, relu=relu, outs=outs)
    assert sc.map_status(m) == 0
    x = wl.feats.cuda()
    for l in range(layers):
        y = sc.subm_forward_packed(m, x, wps[l], relu=relu[l])
        assert torch.equal(fused[l], y), l
        x = y
    # two alternating buffers (the default) give the same final layer
    again = sc.subm_forward_layers(m, wl.feats.cuda(), wps, relu=relu)
    assert torch.equal(again[-1], fused[-1])


def test_fused_stage_six_layers_every_row():
    """The stage workload's six layers (ReLU between them) in one launch: every row of every
    layer against the oracle, each layer fed the GPU's input to it."""
    wl = S.make_workload("stage")
    m = build(wl)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    wps = [sc.wpack_create(w.cuda()) for w in wl.weights]
    L = len(wps)
    relu = [l + 1 < L for l in range(L)]
    outs = [torch.empty((wl.n, wl.c_out), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    ys = sc.subm_forward_layers(m, wl.feats.cuda(), wps, relu=relu, outs=outs)
    assert sc.map_status(m) == 0
    x = wl.feats
    for l in range(L):
        ref = oracle.epilogue_f64(oracle.conv_f64(nbr, x.double().numpy(), wl.weights[l].double().numpy()),
                                  relu=relu[l])
        check_bf16(ys[l], ref)
        x = ys[l].cpu()


def test_fused_layers_errors():
    wl = S.random_cloud(911, 800, shape=(12, 12, 12), c_in=64, c_out=64)
    f = wl.feats.cuda()
    wp = sc.wpack_create(wl.weights[0].cuda())
    wp2 = sc.wpack_create(torch.zeros((27, 64, 32), dtype=torch.bfloat16, device="cuda"))
    m = build(wl)
    with pytest.raises(sc.SpconvError) as e:                    # c_in != c_out in a stack
        sc.subm_forward_layers(m, f, [wp2, wp2])
    assert e.value.code == -1
    mt = build(wl, gemm="tap_major")
    with pytest.raises(sc.SpconvError) as e:                    # only the tile-union GEMM stacks
        sc.subm_forward_layers(mt, f, [wp, wp])
    assert e.value.code == -2
    ms = sc.build_map_strided(wl.coords.cuda(), wl.spatial_shape, 1)
    with pytest.raises(sc.SpconvError) as e:                    # a strided map's rows are not its inputs
        sc.subm_forward_layers(ms, f, [wp, wp])
    assert e.value.code in (-1, -2)
    buf = torch.empty((wl.n, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sc.SpconvError) as e:                    # a layer's output overlaps its input
        sc.subm_forward_layers(m, f, [wp, wp], outs=[buf, buf])
    assert e.value.code == -7
    assert sc.map_status(m) == 0
