"""Pins of the CPU oracle against things other than itself.

Each check below fixes the oracle to something independent: a hand-derived
worked example, closed forms on a dense cube, brute-force all-pairs search,
a library dense convolution (torch ``conv3d`` with padding 1, fp64, CPU) on a
zero-filled grid, and invariants of the definition.  The mutation tests plant
plausible mistakes in copies of the oracle's output (or feed it a mistaken
input) and show that the pins catch them.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from submanifold_sparse_convolution_gb300 import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tap_of(dx, dy, dz):
    return 9 * (dx + 1) + 3 * (dy + 1) + (dz + 1)


OFFSETS = [(dx, dy, dz) for dx in (-1, 0, 1) for dy in (-1, 0, 1) for dz in (-1, 0, 1)]


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            vals[key] = [int(v) for v in rest]
    return vals


# ---------------------------------------------------------------------------
# independent checkers
# ---------------------------------------------------------------------------

def brute_force_nbr(coords):
    """All-pairs search: j is the tap-k neighbour of i iff c[j] - c[i] == d_k, same b."""
    c = np.asarray(coords, dtype=np.int64)
    n = c.shape[0]
    nbr = np.full((n, 27), -1, dtype=np.int64)
    diff = c[None, :, :] - c[:, None, :]          # [i, j, 4]
    same_b = diff[:, :, 0] == 0
    for k, (dx, dy, dz) in enumerate(OFFSETS):
        hit = same_b & (diff[:, :, 1] == dx) & (diff[:, :, 2] == dy) & (diff[:, :, 3] == dz)
        i_idx, j_idx = np.nonzero(hit)
        nbr[i_idx, k] = j_idx
    return nbr


def dense_conv_reference(coords, shape, batch, feats, weights):
    """torch conv3d (padding 1, fp64) on a zero-filled dense grid, read at active sites."""
    X, Y, Z = shape
    f = torch.as_tensor(np.asarray(feats, dtype=np.float64))
    w = torch.as_tensor(np.asarray(weights, dtype=np.float64))   # [27, Cin, Cout]
    c_in, c_out = w.shape[1], w.shape[2]
    grid = torch.zeros(batch, c_in, X, Y, Z, dtype=torch.float64)
    c = torch.as_tensor(np.asarray(coords, dtype=np.int64))
    grid[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]] = f
    wd = torch.zeros(c_out, c_in, 3, 3, 3, dtype=torch.float64)
    for k, (dx, dy, dz) in enumerate(OFFSETS):
        wd[:, :, dx + 1, dy + 1, dz + 1] = w[k].T
    out = torch.nn.functional.conv3d(grid, wd, padding=1)
    return out[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]].numpy()


def pairs_cover_map(nbr, tap_off, in_rows, out_rows):
    """Full-tap coverage: per tap, the pair set equals {(nbr[i][k], i)}."""
    for k in range(27):
        seg = slice(tap_off[k], tap_off[k + 1])
        got = set(zip(in_rows[seg].tolist(), out_rows[seg].tolist()))
        rows = np.nonzero(nbr[:, k] >= 0)[0]
        want = set(zip(nbr[rows, k].tolist(), rows.tolist()))
        if got != want or len(got) != tap_off[k + 1] - tap_off[k]:
            return False
    return True


def pairs_follow_perm(perm, tap_off, out_rows):
    """Within each tap the pairs appear in the order of ``perm``."""
    pos = np.empty_like(perm)
    pos[perm] = np.arange(perm.shape[0])
    for k in range(27):
        s = pos[out_rows[tap_off[k]:tap_off[k + 1]]]
        if np.any(np.diff(s) <= 0):
            return False
    return True


# ---------------------------------------------------------------------------
# worked example and closed forms
# ---------------------------------------------------------------------------

def test_golden_line_and_isolated():
    g = read_golden("line_and_isolated.txt")
    coords = np.array(g["coords"], dtype=np.int32).reshape(-1, 4)
    feats = np.array(g["feats"], dtype=np.float64).reshape(-1, 1)
    weights = (np.arange(27, dtype=np.float64) + 1).reshape(27, 1, 1)
    res = oracle.subm_conv(coords, g["shape"], g["batch"][0], feats, weights)
    assert res["out"][:, 0].tolist() == g["out"]
    assert res["mask"].tolist() == g["masks"]
    assert int(res["tap_off"][27]) == g["pairs"][0]


def test_dense_cube_closed_forms():
    """A fully occupied 3x3x3 cube: counts factor over the axes."""
    cells = np.array([(0, x, y, z) for x in range(3) for y in range(3) for z in range(3)],
                     dtype=np.int32)
    nbr = oracle.kernel_map(cells, (3, 3, 3), 1)
    per_axis = {0: 2, 1: 3, 2: 2}
    for i, (_, x, y, z) in enumerate(cells):
        assert (nbr[i] >= 0).sum() == per_axis[x] * per_axis[y] * per_axis[z]
    assert (nbr >= 0).sum() == 7 ** 3
    centre = [i for i, c in enumerate(cells.tolist()) if c[1:] == [1, 1, 1]][0]
    assert oracle.masks(nbr)[centre] == (1 << 27) - 1


# ---------------------------------------------------------------------------
# kernel map
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,n,shape,batch", [(1, 200, (8, 8, 8), 1), (2, 600, (10, 9, 7), 3),
                                                (3, 1500, (16, 16, 16), 2), (4, 1, (4, 4, 4), 1),
                                                (5, 512, (8, 8, 8), 1)])
def test_kernel_map_matches_brute_force(seed, n, shape, batch):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch)
    nbr = oracle.kernel_map(wl.coords.numpy(), shape, batch)
    assert np.array_equal(nbr, brute_force_nbr(wl.coords.numpy()))


def test_tiny_workload_kernel_map_matches_brute_force():
    wl = S.make_workload("tiny")
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, wl.batch_size)
    assert np.array_equal(nbr, brute_force_nbr(wl.coords.numpy()))


def test_kernel_map_invariants():
    wl = S.random_cloud(11, 3000, shape=(20, 20, 20), batch_size=2)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 2)
    n = nbr.shape[0]
    assert np.array_equal(nbr[:, 13], np.arange(n))             # centre tap is the row itself
    for k in range(27):                                           # symmetry
        rows = np.nonzero(nbr[:, k] >= 0)[0]
        assert np.array_equal(nbr[nbr[rows, k], 26 - k], rows)
    assert (nbr >= 0).sum() >= n


def test_isolated_voxel_sees_only_centre():
    coords = np.array([[0, 0, 0, 0], [0, 5, 5, 5], [0, 2, 2, 2], [1, 3, 3, 3]], dtype=np.int32)
    nbr = oracle.kernel_map(coords, (8, 8, 8), 2)
    assert np.array_equal(oracle.masks(nbr), np.full(4, 1 << 13, dtype=np.uint32))


def test_batches_never_neighbour():
    coords = np.array([[0, 1, 1, 1], [1, 1, 1, 2], [1, 1, 1, 1]], dtype=np.int32)
    nbr = oracle.kernel_map(coords, (4, 4, 4), 2)
    assert nbr[0].tolist().count(-1) == 26
    assert nbr[1, tap_of(0, 0, -1)] == 2 and nbr[2, tap_of(0, 0, 1)] == 1


def test_kernel_map_errors():
    dup = np.array([[0, 1, 1, 1], [0, 2, 2, 2], [0, 1, 1, 1]], dtype=np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.kernel_map(dup, (4, 4, 4), 1)
    assert e.value.code == oracle.ERR_DUPLICATE
    for bad in ([0, 4, 0, 0], [0, -1, 0, 0], [1, 0, 0, 0], [0, 0, 0, 9]):
        with pytest.raises(oracle.OracleError) as e:
            oracle.kernel_map(np.array([[0, 0, 0, 0], bad], dtype=np.int32), (4, 4, 9), 1)
        assert e.value.code == oracle.ERR_RANGE


def test_mutated_kernel_map_is_caught():
    wl = S.random_cloud(21, 400, shape=(8, 8, 8))
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    ref = brute_force_nbr(wl.coords.numpy())
    bad = nbr.copy()
    bad[:, [tap_of(-1, 0, 0), tap_of(1, 0, 0)]] = bad[:, [tap_of(1, 0, 0), tap_of(-1, 0, 0)]]
    assert not np.array_equal(bad, ref)                           # a swapped offset sign
    bad = nbr.copy()
    bad[:, [tap_of(0, -1, 0), tap_of(-1, 0, 0)]] = bad[:, [tap_of(-1, 0, 0), tap_of(0, -1, 0)]]
    assert not np.array_equal(bad, ref)                           # transposed axes


# ---------------------------------------------------------------------------
# masks, order and pair lists
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("calibrated", [False, True])
def test_order_and_pair_lists(calibrated):
    wl = S.random_cloud(31, 2500, shape=(16, 16, 16), batch_size=2)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 2)
    m = oracle.masks(nbr)
    assert np.array_equal(m, ((nbr >= 0) * (1 << np.arange(27))).sum(1).astype(np.uint32))
    order = oracle.tap_order(m, calibrated)
    assert sorted(order.tolist()) == list(range(27))
    counts = np.array([((m >> t) & 1).sum() for t in range(27)], dtype=np.int64)
    if calibrated:
        assert np.all(np.diff(counts[order]) <= 0)
    else:
        assert order.tolist() == list(range(27))
    key = oracle.sort_keys(m, order)
    popc = lambda a: np.array([bin(int(v)).count("1") for v in a])
    assert np.array_equal(popc(key), popc(m))
    if not calibrated:
        assert np.array_equal(key, m)
    p = oracle.perm(key)
    assert sorted(p.tolist()) == list(range(len(p)))
    ks = key[p]
    assert np.all(np.diff(ks.astype(np.int64)) >= 0)
    ties = np.diff(ks.astype(np.int64)) == 0
    assert np.all(np.diff(p)[ties] > 0)                           # stable: ties by row
    tap_off, ins, outs = oracle.pair_lists(nbr, p)
    assert tap_off[0] == 0 and tap_off[27] == (nbr >= 0).sum()
    assert np.all(np.diff(tap_off) == (nbr >= 0).sum(0))
    assert pairs_cover_map(nbr, tap_off, ins, outs)
    assert pairs_follow_perm(p, tap_off, outs)


def test_calibrated_key_compares_rows_rarest_tap_first():
    # "Calibrated bit order" (Sparse convolution in FP32): taps ranked by descending
    # frequency, the rarest in the most significant key bit.  Restated independently:
    # the tap order is a lexsort of (-count, tap), and two rows compare like their
    # tap sets read from the rarest tap to the commonest, the first difference deciding.
    wl = S.random_cloud(33, 1800, shape=(14, 14, 14), batch_size=1)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    m = oracle.masks(nbr).astype(np.int64)
    counts = (nbr >= 0).sum(0)
    order = oracle.tap_order(oracle.masks(nbr), True)
    assert order.tolist() == np.lexsort((np.arange(27), -counts)).tolist()
    key = oracle.sort_keys(oracle.masks(nbr), order).astype(np.int64)
    rng = np.random.default_rng(34)
    rare_first = order[::-1].tolist()
    for i, j in rng.integers(0, len(m), size=(3000, 2)):
        expect = 0
        for tap in rare_first:
            a, b = (m[i] >> tap) & 1, (m[j] >> tap) & 1
            if a != b:
                expect = 1 if a > b else -1
                break
        assert np.sign(key[i] - key[j]) == expect


def test_mutated_pair_lists_are_caught():
    wl = S.random_cloud(32, 800, shape=(10, 10, 10))
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    p = oracle.perm(oracle.sort_keys(oracle.masks(nbr), oracle.tap_order(oracle.masks(nbr))))
    tap_off, ins, outs = oracle.pair_lists(nbr, p)
    # drop one pair (the mutation the pages use to show their coverage test bites)
    k = 5
    drop = tap_off[k] + 1
    ins2, outs2 = np.delete(ins, drop), np.delete(outs, drop)
    off2 = tap_off.copy()
    off2[k + 1:] -= 1
    assert not pairs_cover_map(nbr, off2, ins2, outs2)
    # swap two pairs inside a tap: coverage holds, order does not
    outs3 = outs.copy()
    outs3[tap_off[k]], outs3[tap_off[k] + 1] = outs3[tap_off[k] + 1], outs3[tap_off[k]]
    assert not pairs_follow_perm(p, tap_off, outs3)


# ---------------------------------------------------------------------------
# features
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed,n,shape,batch,c_in,c_out",
                         [(41, 300, (9, 8, 7), 2, 5, 3), (42, 900, (12, 12, 12), 1, 16, 16),
                          (43, 60, (5, 5, 5), 3, 1, 7)])
def test_conv_matches_dense_conv3d(seed, n, shape, batch, c_in, c_out):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch, c_in=c_in, c_out=c_out)
    nbr = oracle.kernel_map(wl.coords.numpy(), shape, batch)
    f = wl.feats.double().numpy()
    w = wl.weights[0].double().numpy()
    got = oracle.conv_f64(nbr, f, w)
    ref = dense_conv_reference(wl.coords.numpy(), shape, batch, f, w)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_mutated_conv_is_caught():
    """Convolution instead of correlation (mirrored taps) and transposed W both fail."""
    wl = S.random_cloud(44, 400, shape=(9, 9, 9), c_in=6, c_out=6)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    f = wl.feats.double().numpy()
    w = wl.weights[0].double().numpy()
    ref = dense_conv_reference(wl.coords.numpy(), wl.spatial_shape, 1, f, w)
    assert not np.allclose(oracle.conv_f64(nbr, f, w[::-1].copy()), ref, atol=1e-6)
    assert not np.allclose(oracle.conv_f64(nbr, f, w.transpose(0, 2, 1).copy()), ref, atol=1e-6)


def test_conv_isolated_voxel_is_centre_tap_product():
    coords = np.array([[0, 1, 1, 1], [0, 6, 6, 6]], dtype=np.int32)
    rng = np.random.default_rng(5)
    f = rng.standard_normal((2, 4))
    w = rng.standard_normal((27, 4, 3))
    out = oracle.conv_f64(oracle.kernel_map(coords, (8, 8, 8), 1), f, w)
    np.testing.assert_allclose(out, f @ w[13], rtol=1e-14)


def test_conv_row_permutation_equivariance():
    wl = S.random_cloud(51, 700, shape=(11, 11, 11), c_in=8, c_out=8)
    c = wl.coords.numpy()
    f = wl.feats.double().numpy()
    w = wl.weights[0].double().numpy()
    out = oracle.conv_f64(oracle.kernel_map(c, wl.spatial_shape, 1), f, w)
    q = np.random.default_rng(52).permutation(c.shape[0])
    out_q = oracle.conv_f64(oracle.kernel_map(c[q], wl.spatial_shape, 1), f[q], w)
    np.testing.assert_allclose(out_q, out[q], rtol=1e-13, atol=1e-13)


def test_conv_linearity_and_batch_isolation():
    wl = S.random_cloud(61, 600, shape=(10, 10, 10), batch_size=2, c_in=4, c_out=5)
    c = wl.coords.numpy()
    nbr = oracle.kernel_map(c, wl.spatial_shape, 2)
    rng = np.random.default_rng(62)
    f1, f2 = rng.standard_normal((2, c.shape[0], 4))
    w1, w2 = rng.standard_normal((2, 27, 4, 5))
    a, b = 0.75, -1.5
    lhs = oracle.conv_f64(nbr, a * f1 + b * f2, w1)
    rhs = a * oracle.conv_f64(nbr, f1, w1) + b * oracle.conv_f64(nbr, f2, w1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(oracle.conv_f64(nbr, f1, w1 + w2),
                               oracle.conv_f64(nbr, f1, w1) + oracle.conv_f64(nbr, f1, w2),
                               rtol=1e-11, atol=1e-11)
    # changing frame 1's features leaves frame 0's outputs unchanged
    f3 = f1.copy()
    f3[c[:, 0] == 1] = rng.standard_normal(((c[:, 0] == 1).sum(), 4))
    o1, o3 = oracle.conv_f64(nbr, f1, w1), oracle.conv_f64(nbr, f3, w1)
    assert np.array_equal(o1[c[:, 0] == 0], o3[c[:, 0] == 0])


def test_conv_row_subset_matches_full():
    wl = S.random_cloud(71, 500, shape=(9, 9, 9), c_in=3, c_out=2)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1)
    f = wl.feats.double().numpy()
    w = wl.weights[0].double().numpy()
    rows = np.array([7, 3, 499, 0, 3], dtype=np.int32)
    assert np.array_equal(oracle.conv_f64(nbr, f, w, rows=rows), oracle.conv_f64(nbr, f, w)[rows])


# ---------------------------------------------------------------------------
# layer epilogue (scale, bias, residual, ReLU)
# ---------------------------------------------------------------------------

def dense_layer_reference(coords, shape, batch, feats, weights, scale, bias, residual, relu):
    """A dense layer through torch on a zero-filled grid (fp64, CPU): conv3d with
    the per-channel scale folded into the weights and its own bias argument,
    plus the residual, then torch's ReLU."""
    w = np.asarray(weights, dtype=np.float64) * np.asarray(scale, dtype=np.float64)[None, None, :]
    X, Y, Z = shape
    f = torch.as_tensor(np.asarray(feats, dtype=np.float64))
    wt = torch.as_tensor(w)
    c_in, c_out = wt.shape[1], wt.shape[2]
    grid = torch.zeros(batch, c_in, X, Y, Z, dtype=torch.float64)
    c = torch.as_tensor(np.asarray(coords, dtype=np.int64))
    grid[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]] = f
    wd = torch.zeros(c_out, c_in, 3, 3, 3, dtype=torch.float64)
    for k, (dx, dy, dz) in enumerate(OFFSETS):
        wd[:, :, dx + 1, dy + 1, dz + 1] = wt[k].T
    out = torch.nn.functional.conv3d(grid, wd, bias=torch.as_tensor(np.asarray(bias, dtype=np.float64)),
                                     padding=1)
    y = out[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]] + torch.as_tensor(np.asarray(residual, dtype=np.float64))
    return (torch.relu(y) if relu else y).numpy()


@pytest.mark.parametrize("relu", [False, True])
def test_epilogue_matches_dense_layer(relu):
    wl = S.random_cloud(81, 500, shape=(9, 8, 10), batch_size=2, c_in=6, c_out=5)
    c = wl.coords.numpy()
    rng = np.random.default_rng(82)
    f = wl.feats.double().numpy()
    w = wl.weights[0].double().numpy()
    scale = rng.uniform(0.5, 2.0, 5)
    bias = rng.standard_normal(5)
    res = rng.standard_normal((c.shape[0], 5))
    nbr = oracle.kernel_map(c, wl.spatial_shape, 2)
    got = oracle.epilogue_f64(oracle.conv_f64(nbr, f, w), scale, bias, res, relu)
    ref = dense_layer_reference(c, wl.spatial_shape, 2, f, w, scale, bias, res, relu)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    if relu:
        assert (got == 0).any() and (got > 0).any()
    # the row subset form reads the residual rows it is given
    rows = np.array([3, 0, 499, 42], dtype=np.int32)
    sub = oracle.epilogue_f64(oracle.conv_f64(nbr, f, w, rows=rows), scale, bias, res, relu, rows=rows)
    np.testing.assert_allclose(sub, got[rows], rtol=1e-13, atol=1e-13)


def test_mutated_epilogue_is_caught():
    """Scaling after the bias, or the ReLU before the residual, both fail the dense layer."""
    wl = S.random_cloud(83, 400, shape=(9, 9, 9), c_in=4, c_out=4)
    c = wl.coords.numpy()
    rng = np.random.default_rng(84)
    f = wl.feats.double().numpy()
    w = wl.weights[0].double().numpy()
    scale, bias = rng.uniform(0.5, 2.0, 4), rng.standard_normal(4)
    res = rng.standard_normal((c.shape[0], 4))
    conv = oracle.conv_f64(oracle.kernel_map(c, wl.spatial_shape, 1), f, w)
    ref = dense_layer_reference(c, wl.spatial_shape, 1, f, w, scale, bias, res, True)
    wrong_order = np.maximum((conv + bias) * scale + res, 0.0)
    relu_first = np.maximum(conv * scale + bias, 0.0) + res
    assert not np.allclose(wrong_order, ref, atol=1e-6)
    assert not np.allclose(relu_first, ref, atol=1e-6)
    np.testing.assert_allclose(oracle.epilogue_f64(conv, scale, bias, res, True), ref, rtol=1e-12, atol=1e-12)


def test_epilogue_identity_and_defaults():
    rng = np.random.default_rng(85)
    conv = rng.standard_normal((7, 3))
    assert np.array_equal(oracle.epilogue_f64(conv), conv)
    assert np.array_equal(oracle.epilogue_f64(conv, relu=True), np.where(conv > 0, conv, 0.0))
    assert np.array_equal(oracle.epilogue_f64(conv, scale=np.ones(3), bias=np.zeros(3)), conv)


# ---------------------------------------------------------------------------
# kernel size 5 and offset groups
# ---------------------------------------------------------------------------

def offsets_k(K):
    r = (K - 1) // 2
    return [(dx, dy, dz) for dx in range(-r, r + 1) for dy in range(-r, r + 1) for dz in range(-r, r + 1)]


def brute_force_nbr_k(coords, K):
    """All-pairs search for a K x K x K kernel (taps in the order of offsets_k)."""
    c = np.asarray(coords, dtype=np.int64)
    n = c.shape[0]
    offs = offsets_k(K)
    nbr = np.full((n, len(offs)), -1, dtype=np.int64)
    diff = c[None, :, :] - c[:, None, :]
    same_b = diff[:, :, 0] == 0
    for k, (dx, dy, dz) in enumerate(offs):
        hit = same_b & (diff[:, :, 1] == dx) & (diff[:, :, 2] == dy) & (diff[:, :, 3] == dz)
        i_idx, j_idx = np.nonzero(hit)
        nbr[i_idx, k] = j_idx
    return nbr


def dense_conv_reference_k(coords, shape, batch, feats, weights, K):
    """torch conv3d (padding (K-1)/2, fp64) on a zero-filled grid, read at active sites."""
    X, Y, Z = shape
    r = (K - 1) // 2
    f = torch.as_tensor(np.asarray(feats, dtype=np.float64))
    w = torch.as_tensor(np.asarray(weights, dtype=np.float64))
    c_in, c_out = w.shape[1], w.shape[2]
    grid = torch.zeros(batch, c_in, X, Y, Z, dtype=torch.float64)
    c = torch.as_tensor(np.asarray(coords, dtype=np.int64))
    grid[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]] = f
    wd = torch.zeros(c_out, c_in, K, K, K, dtype=torch.float64)
    for k, (dx, dy, dz) in enumerate(offsets_k(K)):
        wd[:, :, dx + r, dy + r, dz + r] = w[k].T
    out = torch.nn.functional.conv3d(grid, wd, padding=r)
    return out[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]].numpy()


def check_group_golden(name):
    g = read_golden(name)
    K, G = g["kernel"][0], g["groups"][0]
    V = K ** 3
    coords = np.array(g["coords"], dtype=np.int32).reshape(-1, 4)
    n = coords.shape[0]
    nbr = oracle.kernel_map(coords, g["shape"], g["batch"][0], K)
    m, _, p = oracle.group_orders(nbr, G)
    assert m.reshape(-1).tolist() == g["masks"]
    assert p.reshape(-1).tolist() == g["perms"]
    tap_off, ins, outs = oracle.pair_lists(nbr, p)
    assert ins.tolist() == g["in_rows"] and outs.tolist() == g["out_rows"]
    counts = np.diff(tap_off)
    want = dict(zip(g["tap_counts"][0::2], g["tap_counts"][1::2]))
    assert counts.tolist() == [want.get(k, 0) for k in range(V)]
    if "out" in g:
        feats = np.array(g["feats"], dtype=np.float64).reshape(-1, 1)
        weights = (np.arange(V, dtype=np.float64) + 1).reshape(V, 1, 1)
        res = oracle.subm_conv(coords, g["shape"], g["batch"][0], feats, weights, kernel_size=K, groups=G)
        assert res["out"][:, 0].tolist() == g["out"]
        assert res["perm"].shape == (G, n)


def test_golden_k3_three_groups():
    check_group_golden("line_k3_three_groups.txt")


def test_golden_k5_five_groups():
    check_group_golden("line_k5_five_groups.txt")


@pytest.mark.parametrize("seed,n,shape,batch", [(91, 300, (9, 8, 7), 2), (92, 700, (10, 10, 10), 1),
                                                (93, 1, (4, 4, 4), 1)])
def test_kernel_map_k5_matches_brute_force(seed, n, shape, batch):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch)
    nbr = oracle.kernel_map(wl.coords.numpy(), shape, batch, 5)
    assert nbr.shape == (n, 125)
    assert np.array_equal(nbr, brute_force_nbr_k(wl.coords.numpy(), 5))


def test_kernel_map_k5_invariants_and_cube():
    wl = S.random_cloud(94, 2000, shape=(14, 14, 14), batch_size=2)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 2, 5)
    n = nbr.shape[0]
    assert np.array_equal(nbr[:, 62], np.arange(n))
    for k in range(125):
        rows = np.nonzero(nbr[:, k] >= 0)[0]
        assert np.array_equal(nbr[nbr[rows, k], 124 - k], rows)
    # the 3x3x3 taps of the 5x5x5 map are the K = 3 map
    nbr3 = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 2, 3)
    inner = [25 * (dx + 2) + 5 * (dy + 2) + (dz + 2) for dx, dy, dz in OFFSETS]
    assert np.array_equal(nbr[:, inner], nbr3)
    # a full 5x5x5 cube: per-axis neighbour counts 3 4 5 4 3, 19^3 pairs
    cells = np.array([(0, x, y, z) for x in range(5) for y in range(5) for z in range(5)], dtype=np.int32)
    cube = oracle.kernel_map(cells, (5, 5, 5), 1, 5)
    per_axis = [3, 4, 5, 4, 3]
    for i, (_, x, y, z) in enumerate(cells):
        assert (cube[i] >= 0).sum() == per_axis[x] * per_axis[y] * per_axis[z]
    assert (cube >= 0).sum() == 19 ** 3


@pytest.mark.parametrize("seed,n,shape,batch,c_in,c_out", [(95, 300, (9, 8, 7), 2, 5, 3),
                                                            (96, 600, (11, 11, 11), 1, 8, 8)])
def test_conv_k5_matches_dense_conv3d(seed, n, shape, batch, c_in, c_out):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch, c_in=c_in, c_out=c_out)
    rng = np.random.default_rng(seed)
    nbr = oracle.kernel_map(wl.coords.numpy(), shape, batch, 5)
    f = wl.feats.double().numpy()
    w = rng.standard_normal((125, c_in, c_out)) * 0.05
    got = oracle.conv_f64(nbr, f, w)
    ref = dense_conv_reference_k(wl.coords.numpy(), shape, batch, f, w, 5)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # a mirrored kernel (convolution instead of correlation) is caught
    assert not np.allclose(oracle.conv_f64(nbr, f, w[::-1].copy()), ref, atol=1e-6)


@pytest.mark.parametrize("K,G", [(3, 3), (5, 5), (3, 1)])
@pytest.mark.parametrize("calibrated", [False, True])
def test_group_orders_and_pair_lists(K, G, calibrated):
    wl = S.random_cloud(97 + K + G, 1500, shape=(13, 13, 13), batch_size=2)
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 2, K)
    V, kg = K ** 3, K ** 3 // G
    m, orders, p = oracle.group_orders(nbr, G, calibrated)
    assert m.shape == (G, nbr.shape[0]) and p.shape == (G, nbr.shape[0])
    present = nbr >= 0
    for g in range(G):
        bits = present[:, g * kg:(g + 1) * kg]
        assert np.array_equal(m[g], (bits * (1 << np.arange(kg, dtype=np.int64))).sum(1).astype(np.uint32))
        counts = bits.sum(0)
        if calibrated:
            assert orders[g].tolist() == np.lexsort((np.arange(kg), -counts)).tolist()
        else:
            assert orders[g].tolist() == list(range(kg))
        key = oracle.sort_keys(m[g], orders[g]).astype(np.int64)
        ks = key[p[g]]
        assert sorted(p[g].tolist()) == list(range(nbr.shape[0]))
        assert np.all(np.diff(ks) >= 0)
        assert np.all(np.diff(p[g])[np.diff(ks) == 0] > 0)
    tap_off, ins, outs = oracle.pair_lists(nbr, p)
    assert tap_off[V] == present.sum() and np.all(np.diff(tap_off) == present.sum(0))
    for k in range(V):
        seg = slice(tap_off[k], tap_off[k + 1])
        got = set(zip(ins[seg].tolist(), outs[seg].tolist()))
        rows = np.nonzero(present[:, k])[0]
        assert got == set(zip(nbr[rows, k].tolist(), rows.tolist()))
        pos = np.empty(nbr.shape[0], dtype=np.int64)
        pos[p[k // kg]] = np.arange(nbr.shape[0])
        assert np.all(np.diff(pos[outs[seg]]) > 0)
    if G == 1:
        # one group is the plain K = 3 order
        assert np.array_equal(p[0], oracle.perm(oracle.sort_keys(oracle.masks(nbr),
                                                                 oracle.tap_order(oracle.masks(nbr), calibrated))))


def test_mutated_group_order_is_caught():
    """Pair lists laid out in one order for all taps (the groups' orders
    ignored) break the property that each tap follows its own group's order."""
    wl = S.random_cloud(99, 1200, shape=(12, 12, 12))
    nbr = oracle.kernel_map(wl.coords.numpy(), wl.spatial_shape, 1, 3)
    _, _, p = oracle.group_orders(nbr, 3)
    tap_off, _, outs = oracle.pair_lists(nbr, p[1])
    pos = np.empty(nbr.shape[0], dtype=np.int64)
    pos[p[0]] = np.arange(nbr.shape[0])
    follows = [np.all(np.diff(pos[outs[tap_off[k]:tap_off[k + 1]]]) > 0) for k in range(9)]
    assert not all(follows)


# ---------------------------------------------------------------------------
# strided convolution (kernel 3, stride 2, padding 1) and its inverse
# ---------------------------------------------------------------------------

def _dense_weights(w):
    """[27, Cin, Cout] taps -> a torch [Cout, Cin, 3, 3, 3] conv3d weight."""
    w = torch.as_tensor(np.asarray(w, dtype=np.float64))
    wd = torch.zeros(w.shape[2], w.shape[1], 3, 3, 3, dtype=torch.float64)
    for k, (dx, dy, dz) in enumerate(OFFSETS):
        wd[:, :, dx + 1, dy + 1, dz + 1] = w[k].T
    return wd


def _grid(coords, values, batch, shape):
    c = torch.as_tensor(np.asarray(coords, dtype=np.int64))
    v = torch.as_tensor(np.asarray(values, dtype=np.float64))
    g = torch.zeros(batch, v.shape[1], *shape, dtype=torch.float64)
    g[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]] = v
    return g


@pytest.mark.parametrize("seed,n,shape,batch", [(111, 300, (9, 8, 7), 2), (112, 800, (12, 12, 12), 1),
                                                (113, 1, (4, 4, 4), 1), (114, 400, (10, 11, 6), 3)])
def test_strided_map_and_conv_match_dense_conv3d(seed, n, shape, batch):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch, c_in=5, c_out=4)
    c = wl.coords.numpy()
    oc, nbr = oracle.strided_map(c, shape, batch)
    oshape = oracle.strided_shape(shape)
    assert oshape == tuple(((np.asarray(shape) + 2 - 3) // 2 + 1).tolist())
    # the output sites are where a stride-2 window holds any input site
    ones = torch.nn.functional.conv3d(_grid(c, np.ones((n, 1)), batch, shape),
                                      torch.ones(1, 1, 3, 3, 3, dtype=torch.float64), stride=2, padding=1)
    assert tuple(ones.shape[2:]) == oshape
    want = np.stack(np.nonzero(ones[:, 0].numpy() > 0), 1).astype(np.int32)   # ascending (b, x, y, z)
    assert np.array_equal(oc, want)
    # values
    f = wl.feats.double().numpy()
    w = np.random.default_rng(seed).standard_normal((27, 5, 4))
    dense = torch.nn.functional.conv3d(_grid(c, f, batch, shape), _dense_weights(w), stride=2, padding=1)
    ref = dense[oc[:, 0], :, oc[:, 1], oc[:, 2], oc[:, 3]].numpy()
    np.testing.assert_allclose(oracle.conv_f64(nbr, f, w), ref, rtol=1e-12, atol=1e-12)
    # every output site has at least one input; the pairs count every (input, window) incidence
    assert (nbr >= 0).any(1).all()
    assert (nbr >= 0).sum() == sum(1 for (b, x, y, z) in c for d in OFFSETS
                                   if all((v - dd) % 2 == 0 and 0 <= (v - dd) // 2 < s
                                          for v, dd, s in zip((x, y, z), d, oshape)))


@pytest.mark.parametrize("seed,n,shape,batch", [(121, 300, (9, 8, 7), 2), (122, 700, (12, 12, 12), 1)])
def test_inverse_map_and_conv_match_dense_conv_transpose3d(seed, n, shape, batch):
    wl = S.random_cloud(seed, n, shape=shape, batch_size=batch)
    c = wl.coords.numpy()
    oc, nbr = oracle.strided_map(c, shape, batch)
    inv = oracle.inverse_map(nbr, n)
    oshape = oracle.strided_shape(shape)
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((oc.shape[0], 3))
    w = rng.standard_normal((27, 3, 6))           # [tap][C_in][C_out] of the inverse convolution
    wt = torch.zeros(3, 6, 3, 3, 3, dtype=torch.float64)   # conv_transpose3d: [C_in, C_out, kx, ky, kz]
    for k, (dx, dy, dz) in enumerate(OFFSETS):
        wt[:, :, dx + 1, dy + 1, dz + 1] = torch.as_tensor(w[k])
    pad = tuple(int(s % 2 == 0) for s in shape)   # output_padding recovers an even extent
    dense = torch.nn.functional.conv_transpose3d(_grid(oc, y, batch, oshape), wt, stride=2, padding=1,
                                                 output_padding=pad)
    assert tuple(dense.shape[2:]) == tuple(shape)
    ref = dense[c[:, 0], :, c[:, 1], c[:, 2], c[:, 3]].numpy()
    np.testing.assert_allclose(oracle.conv_f64(inv, y, w), ref, rtol=1e-12, atol=1e-12)
    # the inverse map is the strided map read backwards
    for o, k in zip(*np.nonzero(nbr >= 0)):
        assert inv[nbr[o, k], k] == o
    assert (inv >= 0).sum() == (nbr >= 0).sum()


def test_golden_strided_and_inverse():
    g = read_golden("line_strided_and_inverse.txt")
    coords = np.array(g["coords"], dtype=np.int32).reshape(-1, 4)
    n = coords.shape[0]
    assert oracle.strided_shape(g["shape"]) == tuple(g["out_shape"])
    oc, nbr = oracle.strided_map(coords, g["shape"], g["batch"][0])
    assert oc.reshape(-1).tolist() == g["out_coords"]
    want = np.full((oc.shape[0], 27), -1, dtype=np.int32)
    for o, k, i in zip(*[iter(g["nbr"])] * 3):
        want[o, k] = i
    assert np.array_equal(nbr, want)
    inv = oracle.inverse_map(nbr, n)
    want_inv = np.full((n, 27), -1, dtype=np.int32)
    for i, k, o in zip(*[iter(g["inv"])] * 3):
        want_inv[i, k] = o
    assert np.array_equal(inv, want_inv)
    w = (np.arange(27, dtype=np.float64) + 1).reshape(27, 1, 1)
    f = np.array(g["feats"], dtype=np.float64).reshape(-1, 1)
    assert oracle.conv_f64(nbr, f, w)[:, 0].tolist() == g["out"]
    y = np.array(g["inv_feats"], dtype=np.float64).reshape(-1, 1)
    assert oracle.conv_f64(inv, y, w)[:, 0].tolist() == g["inv_out"]


def test_mutated_strided_map_is_caught():
    """Windows at o + d (no stride) or at 2o - d (mirrored) both fail the dense conv."""
    wl = S.random_cloud(131, 500, shape=(10, 10, 10), c_in=3, c_out=3)
    c = wl.coords.numpy()
    oc, nbr = oracle.strided_map(c, (10, 10, 10), 1)
    f = wl.feats.double().numpy()
    w = np.random.default_rng(132).standard_normal((27, 3, 3))
    dense = torch.nn.functional.conv3d(_grid(c, f, 1, (10, 10, 10)), _dense_weights(w), stride=2, padding=1)
    ref = dense[oc[:, 0], :, oc[:, 1], oc[:, 2], oc[:, 3]].numpy()
    assert not np.allclose(oracle.conv_f64(nbr[:, ::-1].copy(), f, w), ref, atol=1e-6)
    where = {tuple(v): i for i, v in enumerate(c.tolist())}
    nbr_plain = np.array([[where.get((o[0], o[1] + dx, o[2] + dy, o[3] + dz), -1) for dx, dy, dz in OFFSETS]
                          for o in oc.tolist()], dtype=np.int32)
    assert not np.allclose(oracle.conv_f64(nbr_plain, f, w), ref, atol=1e-6)
