"""The seeded workloads have the documented sizes, ranges and uniqueness."""
import numpy as np
import pytest

from submanifold_sparse_convolution_gb300 import synthetic as S

EXPECT = {"tiny": (2000, (32, 32, 32), 1, 16, 16, 1), "outdoor": (32371, (1440, 1440, 40), 1, 128, 128, 1),
          "deep": (15052, (180, 180, 41), 1, 512, 512, 1), "large": (94517, (2095, 2095, 695), 1, 128, 128, 1),
          "stage": (240000, (1440, 1440, 40), 2, 64, 64, 6)}


@pytest.mark.parametrize("name", ["tiny", "outdoor", "deep", "large", "stage"])
def test_workload_shape(name):
    n, shape, batch, cin, cout, layers = EXPECT[name]
    c, sh, b, _ = S.make_coords(name)
    assert c.shape == (n, 4) and c.dtype == np.int32 and tuple(sh) == shape and b == batch
    assert c[:, 0].min() >= 0 and c[:, 0].max() < batch
    for a in range(3):
        assert c[:, a + 1].min() >= 0 and c[:, a + 1].max() < shape[a]
    lin = ((c[:, 0].astype(np.int64) * shape[0] + c[:, 1]) * shape[1] + c[:, 2]) * shape[2] + c[:, 3]
    assert np.unique(lin).shape[0] == n
    c2, _, _, _ = S.make_coords(name)
    assert np.array_equal(c, c2)                     # seeded


def test_large_spans_grid_beyond_int32():
    c, sh, _, _ = S.make_coords("large")
    vol = (sh[0] + 2) * (sh[1] + 2) * (sh[2] + 2)
    assert vol > 2 ** 31
    assert c[:, 1].max() - c[:, 1].min() > 2000 and c[:, 3].max() - c[:, 3].min() > 600


def test_features_and_weights():
    wl = S.make_workload("tiny")
    assert wl.feats.shape == (2000, 16) and str(wl.feats.dtype) == "torch.bfloat16"
    w = wl.weights[0].float()
    assert w.shape == (27, 16, 16)
    assert abs(float(w.std()) - S.weights_std(16)) < 0.1 * S.weights_std(16)
    assert abs(float(wl.feats.float().std()) - 1.0) < 0.05
