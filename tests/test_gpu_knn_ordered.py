"""Parity of the spatially ordered brute-force kNN with the oracle.

Clouds of at least 16384 references with 4096 or more queries and
2 <= k <= 32 are put in cell-code order before the lane kernel runs (the
keys keep the original indices).  These cases cover that path: the query
set equal to the reference set and distinct from it, several clouds, valid
lengths (rows past a query length, fewer valid references than k), exact
ties from coordinates on a coarse grid and duplicated points, and points far
outside the frame the cell codes are taken over.
"""
import numpy as np
import pytest
import torch

import oracle
import point_cloud_neighbor_gb300 as pc

pytestmark = pytest.mark.gpu

THREADS = oracle.default_threads()


def dev():
    return torch.device("cuda:0")


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def grid_cloud(rng, B, n, step=1.0 / 64):
    """Uniform points on a grid of spacing `step`, 2% of them duplicated."""
    x = (rng.integers(0, int(1 / step), size=(B, n, 3)) * step).astype(np.float32)
    dup = rng.choice(n, size=n // 50, replace=False)
    x[:, dup] = x[:, rng.choice(n, size=n // 50)]
    return x


def compare(got_d, got_i, want_d, want_i, what):
    got_i = got_i.reshape(want_i.shape)
    got_d = got_d.reshape(want_d.shape)
    bad = int((got_i != want_i).sum())
    assert bad == 0, f"{what}: {bad} of {want_i.size} indices differ"
    badd = int((got_d.view(np.uint32) != want_d.view(np.uint32)).sum())
    assert badd == 0, f"{what}: {badd} of {want_d.size} distances differ"


@pytest.fixture(autouse=True)
def clean_status():
    yield
    assert pc.pc_device_status(reset=True) == 0


@pytest.mark.parametrize("k", [2, 16, 17, 32])
def test_ordered_self_knn_with_ties(k):
    rng = np.random.default_rng(100 + k)
    x = grid_cloud(rng, 2, 16384)
    d, i = pc.pc_knn(to_dev(x), to_dev(x), k)
    wd, wi = oracle.knn(x, x, k, threads=THREADS)     # every row
    compare(d.cpu().numpy().reshape(-1, k), i.cpu().numpy().reshape(-1, k),
            wd, wi, f"ordered self kNN k={k}")


def test_ordered_distinct_queries_with_lengths_and_outliers():
    rng = np.random.default_rng(7)
    B, Q, N, k = 3, 5000, 20000, 8
    x = grid_cloud(rng, B, N, step=1.0 / 128)
    q = rng.random((B, Q, 3), dtype=np.float32)
    q[0, :50] *= 40.0          # queries far outside the references' frame
    x[1, 5:9] = [-1e6, 3e5, 7.0]  # references far outside too
    ql = np.array([Q, 4321, 4096], dtype=np.int64)
    rl = np.array([N, 17000, 6], dtype=np.int64)   # cloud 2: fewer than k
    d, i = pc.pc_knn(to_dev(q), to_dev(x), k, query_lengths=to_dev(ql),
                     ref_lengths=to_dev(rl))
    wd, wi = oracle.knn_masked(q, x, k, ql, rl, threads=THREADS)
    compare(d.cpu().numpy(), i.cpu().numpy(), wd, wi, "ordered masked kNN")


def test_ordered_squared_and_sqrt_agree():
    rng = np.random.default_rng(9)
    x = rng.random((1, 20000, 3), dtype=np.float32)
    q = rng.random((1, 4096, 3), dtype=np.float32)
    d, i = pc.pc_knn(to_dev(q), to_dev(x), 5)
    s, j = pc.pc_knn(to_dev(q), to_dev(x), 5, squared=True)
    assert torch.equal(i, j)
    assert torch.equal(d, torch.sqrt(s))
    wd, wi = oracle.knn(q, x, 5, threads=THREADS)
    compare(d.cpu().numpy().reshape(-1, 5), i.cpu().numpy().reshape(-1, 5),
            wd, wi, "ordered kNN distinct queries")


def test_sm_reserve_only_changes_the_plan():
    rng = np.random.default_rng(11)
    x = to_dev(rng.random((1, 30000, 3), dtype=np.float32))
    n = pc.pc_fps_sm_count(1, 30000, 4096)
    assert 1 <= n <= torch.cuda.get_device_properties(0).multi_processor_count
    d0, i0 = pc.pc_knn(x, x, 12)
    b0, j0 = pc.pc_ball_query(x, x, 0.05, 24)
    try:
        for reserve in (n, 100, 10_000):
            pc.pc_set_sm_reserve(reserve)
            d1, i1 = pc.pc_knn(x, x, 12)
            assert torch.equal(i0, i1) and torch.equal(d0, d1), reserve
            b1, j1 = pc.pc_ball_query(x, x, 0.05, 24)
            assert torch.equal(j0, j1) and torch.equal(b0, b1), reserve
    finally:
        pc.pc_set_sm_reserve(0)


@pytest.mark.parametrize("k", [4, 16])
def test_ordered_unit_plans_agree(k):
    """The launch splits the queries into blocks of 32-query units; SM counts
    that make the units per block odd leave warps with one query per lane.
    Every plan gives the oracle's result, on a ragged query count."""
    rng = np.random.default_rng(23 + k)
    x = grid_cloud(rng, 1, 16384, step=1.0 / 96)
    q = rng.random((1, 4133, 3), dtype=np.float32)
    q[0, :200] = x[0, rng.choice(16384, 200, replace=False)]  # exact matches
    wd, wi = oracle.knn(q, x, k, threads=THREADS)
    qd, xd = to_dev(q), to_dev(x)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    try:
        for reserve in (0, sms - 92, sms - 12, sms - 1):
            pc.pc_set_sm_reserve(max(0, reserve))
            d, i = pc.pc_knn(qd, xd, k)
            compare(d.cpu().numpy(), i.cpu().numpy(), wd, wi,
                    f"ordered kNN k={k}, reserve {reserve}")
    finally:
        pc.pc_set_sm_reserve(0)
