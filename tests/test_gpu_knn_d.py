"""GPU parity of the D-dimensional kNN (dimension-by-dimension distance).

Indices and distances bit-identical to the oracle: same operation order per
pair, same (s, j) total order.  Lattice inputs force exact ties; D = 3 must
equal the point operator; the DGCNN EdgeConv feature shape (1024 points,
64 dimensions, k = 20) is compared in full.
"""
import numpy as np
import pytest
import torch

import oracle
import point_cloud_neighbor_gb300 as pc
from test_gpu_parity import THREADS, assert_dist_equal, assert_idx_equal, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_status():
    yield
    assert pc.pc_device_status(reset=True) == 0


def feats(seed, B, N, D, lattice=None):
    rng = np.random.default_rng(seed)
    if lattice:
        return (rng.integers(0, lattice, (B, N, D)) / lattice).astype(np.float32)
    return rng.standard_normal((B, N, D)).astype(np.float32)


def check(q, x, k, squared=False, what="knn_d"):
    d, i = pc.pc_knn_d(to_dev(q), to_dev(x), k, squared=squared)
    wd, wi = oracle.knn_d(q, x, k, squared=squared, threads=THREADS)
    assert_idx_equal(i.cpu().numpy().reshape(-1, k), wi, what)
    assert_dist_equal(d.cpu().numpy().reshape(-1, k), wd, what)


@pytest.mark.parametrize("B,Q,N,D,k,lattice", [
    (1, 1, 1, 1, 1, None), (2, 65, 300, 7, 20, 4), (3, 130, 1000, 64, 32, None),
    (1, 64, 33, 256, 32, 2), (2, 200, 1024, 17, 5, None), (1, 70, 97, 5, 32, 3),
    (2, 33, 40, 128, 1, None),
])
def test_knn_d_matches_oracle(B, Q, N, D, k, lattice):
    q = feats(10 + D, B, Q, D, lattice)
    x = feats(20 + D, B, N, D, lattice)
    check(q, x, k, what=f"knn_d B={B} Q={Q} N={N} D={D} k={k}")
    check(q, x, k, squared=True, what="knn_d squared")


def test_knn_d_three_dimensions_equals_point_knn():
    rng = np.random.default_rng(30)
    x = rng.random((2, 3000, 3), dtype=np.float32)
    q = rng.random((2, 500, 3), dtype=np.float32)
    d, i = pc.pc_knn_d(to_dev(q), to_dev(x), 16)
    d3, i3 = pc.pc_knn(to_dev(q), to_dev(x), 16)
    assert torch.equal(i, i3)
    assert torch.equal(d.view(torch.int32), d3.view(torch.int32))


def test_knn_d_dgcnn_feature_shape():
    # DGCNN EdgeConv: every point's 20 nearest neighbours in a 64-d feature space
    x = feats(31, 4, 1024, 64)
    check(x, x, 20, what="knn_d DGCNN shape")


def test_knn_d_limits():
    x = to_dev(feats(32, 1, 50, 8))
    with pytest.raises(pc.PointCloudError) as e:
        pc.pc_knn_d(x, x, 33)
    assert e.value.status == 2
    big = to_dev(feats(33, 1, 50, 257))
    with pytest.raises(pc.PointCloudError) as e:
        pc.pc_knn_d(big, big, 4)
    assert e.value.status == 2
    with pytest.raises(pc.PointCloudError):
        pc.pc_knn_d(x, x, 51)


@pytest.mark.parametrize("offset", [1e3, 1e5])
@pytest.mark.parametrize("D", [16, 64, 128])
def test_knn_d_translated_features(offset, D):
    """Features far from the origin (each squared difference rounds at a
    larger exponent): every row the oracle's."""
    x = (feats(40 + D, 2, 700, D).astype(np.float64) + offset).astype(np.float32)
    q = (feats(50 + D, 2, 130, D).astype(np.float64) + offset).astype(np.float32)
    check(q, x, 20, what=f"knn_d +{offset:g} D={D}")


def test_knn_d_zero_dimension_changes_nothing():
    """One more dimension that is zero in every row adds +0 to every s: the
    same indices and bit-identical distances."""
    x = feats(60, 2, 900, 128)
    q = feats(61, 2, 200, 128)
    d1, i1 = pc.pc_knn_d(to_dev(q), to_dev(x), 24)
    pad = lambda a: np.concatenate([a, np.zeros(a.shape[:2] + (1,), np.float32)], axis=2)
    d2, i2 = pc.pc_knn_d(to_dev(pad(q)), to_dev(pad(x)), 24)
    assert torch.equal(i1, i2)
    assert torch.equal(d1.view(torch.int32), d2.view(torch.int32))


def test_knn_d_huge_and_infinite_features():
    """Coordinates near the float range (squares up to ~1e32) and an
    infinite one: the exact s decides as in the oracle (the contract covers
    finite inputs; an infinite s sorts last, ties by index)."""
    x = feats(70, 1, 600, 32)
    q = feats(71, 1, 100, 32)
    x[0, 17, :] = 3e15
    x[0, 40, 0] = np.inf
    x[0, 41, :] = -2e15
    q[0, 9, :] = 2e15
    q[0, 10, :5] = 1e16
    check(q, x, 16, what="knn_d huge and infinite")
