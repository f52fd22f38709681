"""Parity of the grid-accelerated kNN and Ball Query with the oracle.

The grid path must return exactly what the brute-force operators return
(same indices, bit-identical distances): it changes which pairs are
examined, never the arithmetic or the order.  Cases stress what a grid can
get wrong: points on cell faces and exact ties (lattice coordinates), a
degenerate extent (all points equal, flat clouds), queries outside the
reference bounding box, very small and very large radii, subnormal
coordinates, misaligned batches and empty reference sets.
"""
import numpy as np
import pytest
import torch

import _oracle_cache as cache
import oracle
import point_cloud_neighbor_gb300 as pc
from point_cloud_neighbor_gb300 import inputs
from test_gpu_parity import (THREADS, assert_dist_equal, assert_idx_equal,
                             bq_row_properties, knn_row_properties, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_status():
    yield
    assert pc.pc_device_status(reset=True) == 0


def grid_knn(q, x, k):
    g = pc.pc_grid_build(to_dev(x))
    d, i = pc.pc_knn_grid(to_dev(q), g, k)
    return d.cpu().numpy().reshape(-1, k), i.cpu().numpy().reshape(-1, k)


def grid_bq(q, x, r, K):
    g = pc.pc_grid_build(to_dev(x))
    d2, i = pc.pc_ball_query_grid(to_dev(q), g, r, K)
    return d2.cpu().numpy().reshape(-1, K), i.cpu().numpy().reshape(-1, K)


def check_grid_knn(q, x, k, rows=None, what="grid knn"):
    d, i = grid_knn(q, x, k)
    wd, wi = oracle.knn(q, x, k, rows=rows, threads=THREADS)
    if rows is not None:
        d, i = d[rows], i[rows]
    assert_idx_equal(i, wi, what)
    assert_dist_equal(d, wd, what)


def check_grid_bq(q, x, r, K, rows=None, what="grid bq"):
    d2, i = grid_bq(q, x, r, K)
    wd2, wi = oracle.ball_query(q, x, r, K, rows=rows, threads=THREADS)
    if rows is not None:
        d2, i = d2[rows], i[rows]
    assert_idx_equal(i, wi, what)
    assert_dist_equal(d2, wd2, what)


def test_grid_tiny_workload():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.tiny()
    c = np.ascontiguousarray(x[:, oracle.fps(x, cfg["npoint"], 0)[0]])
    check_grid_knn(c, x, cfg["knn_k"], what="grid knn tiny")
    check_grid_bq(c, x, 0.125, 16, what="grid bq tiny")
    check_grid_knn(x, x, 16, what="grid knn tiny all points")


def test_grid_point_mae_and_pointnet2():
    x = inputs.point_mae()
    c = np.ascontiguousarray(np.take_along_axis(
        x, oracle.fps(x, 512, 0, threads=THREADS)[..., None], axis=1))
    check_grid_knn(c, x, 32, what="grid knn point_mae")
    x3 = inputs.pointnet2()
    c3 = np.ascontiguousarray(np.take_along_axis(
        x3, oracle.fps(x3, 1024, 0, threads=THREADS)[..., None], axis=1))
    check_grid_bq(c3, x3, 0.1, 32, what="grid bq pointnet2 r=0.1")
    check_grid_bq(c3, x3, 0.2, 64, what="grid bq pointnet2 r=0.2")
    check_grid_knn(x3, c3, 3, what="grid knn three_nn")


@pytest.mark.slow
@pytest.mark.parametrize("morton", [False, True], ids=["random", "morton"])
def test_grid_large_full(morton):
    """Grid kNN k=16 and Ball Query r=0.02 K=32 over the 100k cloud: every
    row against the oracle, and equal to the brute-force kernels."""
    x = cache.large(morton)
    xd = to_dev(x)
    g = pc.pc_grid_build(xd)
    d, i = pc.pc_knn_grid(xd, g, 16)
    d2, i2 = pc.pc_ball_query_grid(xd, g, 0.02, 32)
    wd, wi = cache.large_knn(morton)
    assert_idx_equal(i.cpu().numpy().reshape(-1, 16), wi, "grid knn large, every row")
    assert_dist_equal(d.cpu().numpy().reshape(-1, 16), wd, "grid knn large, every row")
    wd2, wi2 = cache.large_ball_query(morton)
    assert_idx_equal(i2.cpu().numpy().reshape(-1, 32), wi2, "grid bq large, every row")
    assert_dist_equal(d2.cpu().numpy().reshape(-1, 32), wd2, "grid bq large, every row")
    bd, bi = pc.pc_knn(xd, xd, 16)
    assert torch.equal(i, bi) and torch.equal(d.view(torch.int32), bd.view(torch.int32))
    bd2, bi2 = pc.pc_ball_query(xd, xd, 0.02, 32)
    assert torch.equal(i2, bi2) and torch.equal(d2.view(torch.int32), bd2.view(torch.int32))


@pytest.mark.slow
def test_grid_very_large_full():
    """Grid kNN k=32 and Ball Query r=0.01 K=64 of the 16,384 FPS centres
    against the 1M-point cloud, every row against the oracle."""
    x, _, q = cache.very_large()
    d, i = grid_knn(q, x, 32)
    wd, wi = cache.very_large_knn()
    assert_idx_equal(i, wi, "grid knn 1M, every row")
    assert_dist_equal(d, wd, "grid knn 1M, every row")
    knn_row_properties(q, x, d, i)
    d2, i2 = grid_bq(q, x, 0.01, 64)
    wd2, wi2 = oracle.ball_query(q, x, 0.01, 64, threads=THREADS)
    assert_idx_equal(i2, wi2, "grid bq 1M, every row")
    assert_dist_equal(d2, wd2, "grid bq 1M, every row")
    bq_row_properties(q, x, 0.01, d2, i2)


@pytest.mark.parametrize("B,Q,N,k", [
    (1, 1, 1, 1), (1, 5, 7, 7), (3, 33, 301, 31), (2, 65, 1001, 33),
    (5, 130, 257, 64), (2, 17, 999, 65), (1, 40, 3000, 128), (2, 9, 700, 256),
])
def test_grid_knn_edge_sizes_lattice(B, Q, N, k):
    x = inputs.random_cloud(700 + N, B, N, grid=1 / 16)
    q = inputs.random_cloud(800 + Q, B, Q, grid=1 / 16)
    check_grid_knn(q, x, k, what=f"grid knn B={B} Q={Q} N={N} k={k}")


@pytest.mark.parametrize("B,Q,N,r,K", [
    (1, 1, 0, 0.5, 4), (2, 7, 0, 0.5, 3), (1, 3, 1, 0.5, 1), (3, 33, 301, 0.4, 31),
    (2, 65, 1001, 0.3, 33), (5, 130, 257, 0.8, 65), (2, 17, 999, 2.5, 16),
    (1, 40, 3000, 0.2, 100), (1, 40, 3000, 0.01, 8), (2, 9, 700, 5.0, 256),
])
def test_grid_ball_query_edge_sizes_lattice(B, Q, N, r, K):
    x = inputs.random_cloud(900 + N, B, N, grid=1 / 16)
    q = inputs.random_cloud(1000 + Q, B, Q, grid=1 / 16)
    check_grid_bq(q, x, r, K, what=f"grid bq B={B} Q={Q} N={N} r={r} K={K}")


def test_grid_random_coordinates_and_outside_queries():
    x = inputs.random_cloud(11, 2, 4000)               # in [-1, 1)^3
    q = (inputs.random_cloud(12, 2, 300) * 3.0).astype(np.float32)  # many outside
    check_grid_knn(q, x, 20, what="grid knn outside queries")
    check_grid_bq(q, x, 0.35, 40, what="grid bq outside queries")


def test_grid_degenerate_extents():
    same = np.ones((1, 500, 3), np.float32)
    check_grid_knn(same[:, :10], same, 12, what="grid knn identical points")
    check_grid_bq(same[:, :10], same, 0.1, 20, what="grid bq identical points")
    flat = inputs.random_cloud(13, 1, 800)
    flat[..., 2] = 0.25                                 # zero extent along z
    check_grid_knn(flat[:, :50], flat, 10, what="grid knn flat cloud")
    line = np.zeros((1, 300, 3), np.float32)
    line[0, :, 0] = np.arange(300, dtype=np.float32)    # exact ties everywhere
    check_grid_knn(line, line, 5, what="grid knn line ties")
    check_grid_bq(line, line, 2.0, 6, what="grid bq line boundary")


def test_grid_subnormal_coordinates():
    x = (inputs.random_cloud(14, 1, 700) * np.float32(1e-21)).astype(np.float32)
    q = (inputs.random_cloud(15, 1, 40) * np.float32(1e-21)).astype(np.float32)
    check_grid_knn(q, x, 20, what="grid knn subnormal")
    check_grid_bq(q, x, 1.2e-21, 30, what="grid bq subnormal")


def test_grid_reused_for_many_queries():
    x = inputs.random_cloud(16, 3, 2001)
    g = pc.pc_grid_build(to_dev(x))
    for seed in range(3):
        q = inputs.random_cloud(17 + seed, 3, 55)
        d, i = pc.pc_knn_grid(to_dev(q), g, 9)
        wd, wi = oracle.knn(q, x, 9)
        assert_idx_equal(i.cpu().numpy().reshape(-1, 9), wi, "grid reuse")
        d2, i2 = pc.pc_ball_query_grid(to_dev(q), g, 0.3, 12)
        wd2, wi2 = oracle.ball_query(q, x, 0.3, 12)
        assert_idx_equal(i2.cpu().numpy().reshape(-1, 12), wi2, "grid reuse bq")


def test_grid_invalid_arguments():
    x = to_dev(inputs.random_cloud(18, 1, 10))
    g = pc.pc_grid_build(x)
    with pytest.raises(pc.PointCloudError):
        pc.pc_knn_grid(x, g, 11)
    with pytest.raises(pc.PointCloudError):
        pc.pc_ball_query_grid(x, g, 0.0, 3)
    with pytest.raises(pc.PointCloudError) as e:
        pc.pc_ball_query_grid(x, g, 0.5, 257)
    assert e.value.status == 2
