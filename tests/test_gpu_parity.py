"""Parity of the CUDA kernels (through the C ABI) with the oracle.

Indices must be identical.  Distances are computed in the same operation
order on both sides ((dx*dx + dy*dy) + dz*dz, round to nearest, no FMA;
correctly rounded sqrt), so they must be bit-identical too -- stricter than
the 1e-6 relative bound the contract allows.  Mismatches are reported as
counts.

Sizes: every workload runs on the GPU at its full size in the same launch
configuration as the benchmark, and the oracle checks every output row,
including all 100,000 kNN and Ball Query rows of the 100k-point cloud (random
and Morton order) and all 16,384 rows of the 1M-point cloud (the kNN ones take
the oracle minutes on the host cores: they are marked slow).  Properties that
hold at any size are checked on every row as a second line.
"""
import numpy as np
import pytest
import torch

import _oracle_cache as cache
import oracle
import point_cloud_neighbor_gb300 as pc
from point_cloud_neighbor_gb300 import inputs

pytestmark = pytest.mark.gpu

THREADS = oracle.default_threads()


def dev():
    return torch.device("cuda:0")


def to_dev(a):
    a = np.ascontiguousarray(a)
    if not a.flags.writeable:       # cached oracle inputs are read-only
        a = a.copy()
    return torch.from_numpy(a).to(dev())


def same_bits(a, b):
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


def assert_idx_equal(got, want, what):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    bad = int((got != want).sum())
    assert bad == 0, f"{what}: {bad} of {got.size} indices differ"


def assert_dist_equal(got, want, what):
    bad = int((np.asarray(got).view(np.uint32) != np.asarray(want).view(np.uint32)).sum())
    assert bad == 0, f"{what}: {bad} of {np.asarray(got).size} distances differ"


@pytest.fixture(autouse=True)
def clean_status():
    yield
    assert pc.pc_device_status(reset=True) == 0


# --------------------------------------------------------------------------
# helpers: run the GPU op, compare with the oracle on all or sampled rows
# --------------------------------------------------------------------------
def gpu_fps(x, npoint, start=0, **kw):
    return pc.pc_fps(to_dev(x), npoint, start, **kw).cpu().numpy()


def gpu_knn(q, x, k):
    d, i = pc.pc_knn(to_dev(q), to_dev(x), k)
    return d.cpu().numpy().reshape(-1, k), i.cpu().numpy().reshape(-1, k)


def gpu_bq(q, x, r, K):
    d2, i = pc.pc_ball_query(to_dev(q), to_dev(x), r, K)
    return d2.cpu().numpy().reshape(-1, K), i.cpu().numpy().reshape(-1, K)


def check_knn(q, x, k, rows=None, what="knn"):
    d, i = gpu_knn(q, x, k)
    wd, wi = oracle.knn(q, x, k, rows=rows, threads=THREADS)
    if rows is not None:
        d, i = d[rows], i[rows]
    assert_idx_equal(i, wi, what)
    assert_dist_equal(d, wd, what)


def check_bq(q, x, r, K, rows=None, what="ball_query"):
    d2, i = gpu_bq(q, x, r, K)
    wd2, wi = oracle.ball_query(q, x, r, K, rows=rows, threads=THREADS)
    if rows is not None:
        d2, i = d2[rows], i[rows]
    assert_idx_equal(i, wi, what)
    assert_dist_equal(d2, wd2, what)
    return d2, i


def knn_row_properties(q, x, d, i):
    """Properties of every kNN row that hold at any size: valid distinct
    indices, strictly increasing (s, j) with s the oracle's s32 of the pair,
    and D the correctly rounded sqrt of s."""
    B, Q, _ = q.shape
    k = i.shape[1]
    N = x.shape[1]
    assert i.min() >= 0 and i.max() < N
    b = np.repeat(np.arange(B), Q * k)
    pts = x[b, i.reshape(-1)]
    qq = np.repeat(q.reshape(-1, 3), k, axis=0)
    s = oracle.s32(qq, pts).reshape(-1, k)
    want_d = np.sqrt(s.astype(np.float64)).astype(np.float32)
    assert_dist_equal(d, want_d, "knn distance = sqrt(s32(query, neighbor))")
    if k > 1:
        inc = (s[:, 1:] > s[:, :-1]) | ((s[:, 1:] == s[:, :-1]) & (i[:, 1:] > i[:, :-1]))
        assert inc.all(), f"{int((~inc).sum())} rows not increasing in (s, j)"


def bq_row_properties(q, x, r, d2, i):
    """Properties of every Ball Query row: hits first in increasing index
    order, then (-1, 0) padding; every hit's s32 equals the returned value
    and is < R2."""
    B, Q, _ = q.shape
    K = i.shape[1]
    R2 = oracle.radius_threshold(r)
    valid = i >= 0
    # padding only after the hits
    assert not (np.diff(valid.astype(np.int8), axis=1) > 0).any()
    assert (d2[~valid] == 0).all()
    # strictly increasing indices among hits
    ii = np.where(valid, i, np.iinfo(np.int64).max)
    assert ((ii[:, 1:] > ii[:, :-1]) | ~valid[:, 1:]).all()
    rows, cols = np.nonzero(valid)
    b = rows // Q
    s = oracle.s32(q.reshape(-1, 3)[rows], x[b, i[rows, cols]])
    assert_dist_equal(d2[rows, cols], s, "ball query distance = s32")
    assert (s < R2).all()


# --------------------------------------------------------------------------
# worked example (project page, "Minimal example")
# --------------------------------------------------------------------------
def test_worked_example():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "worked_example.json")))
    xyz = np.array(g["xyz"], np.float32)
    idx = gpu_fps(xyz, 2, 0)
    assert idx.tolist() == g["fps"]["idx"]
    centers = np.ascontiguousarray(xyz[:, idx[0]])
    d, i = gpu_knn(centers, xyz, 2)
    assert i.reshape(1, 2, 2).tolist() == g["knn"]["idx"]
    assert d.reshape(1, 2, 2).tolist() == g["knn"]["dist"]
    d2, i2 = gpu_bq(centers, xyz, 1.1, 2)
    assert i2.reshape(1, 2, 2).tolist() == g["ball_query"]["idx"]
    assert d2.reshape(1, 2, 2).tolist() == g["ball_query"]["dist2"]


# --------------------------------------------------------------------------
# workload 1: tiny, exact ties on the 1/64 grid
# --------------------------------------------------------------------------
def test_tiny_all_ops_full():
    cfg = inputs.CONFIGS["tiny"]
    x = inputs.tiny()
    idx = gpu_fps(x, cfg["npoint"], 0)
    want = oracle.fps(x, cfg["npoint"], 0)
    assert_idx_equal(idx, want, "fps tiny")
    centers = np.ascontiguousarray(x[:, want[0]])
    check_knn(centers, x, cfg["knn_k"], what="knn tiny")
    for r, K in cfg["bq"]:
        check_bq(centers, x, r, K, what="bq tiny")


# --------------------------------------------------------------------------
# workload 2: Point-MAE grouping, B=32 x 8192, FPS 512, kNN k=32
# --------------------------------------------------------------------------
def test_point_mae_full():
    cfg = inputs.CONFIGS["point_mae"]
    x = inputs.point_mae()
    idx = gpu_fps(x, cfg["npoint"], 0)
    want = oracle.fps(x, cfg["npoint"], 0, threads=THREADS)
    assert_idx_equal(idx, want, "fps point_mae")
    centers = np.ascontiguousarray(np.take_along_axis(x, want[..., None], axis=1))
    check_knn(centers, x, cfg["knn_k"], what="knn point_mae")


# --------------------------------------------------------------------------
# workload 3: PointNet++ set abstraction, B=16 x 4096
# --------------------------------------------------------------------------
def test_pointnet2_full():
    cfg = inputs.CONFIGS["pointnet2"]
    x = inputs.pointnet2()
    idx = gpu_fps(x, cfg["npoint"], 0)
    want = oracle.fps(x, cfg["npoint"], 0, threads=THREADS)
    assert_idx_equal(idx, want, "fps pointnet2")
    centers = np.ascontiguousarray(np.take_along_axis(x, want[..., None], axis=1))
    for r, K in cfg["bq"]:
        check_bq(centers, x, r, K, what=f"bq pointnet2 r={r}")
    # three_nn shape: every point queries its 3 nearest centers
    check_knn(x, centers, cfg["knn_k"], what="knn pointnet2 three_nn")


# --------------------------------------------------------------------------
# workload 4: one 100k-point cloud, random order and Morton-sorted
# --------------------------------------------------------------------------
@pytest.mark.parametrize("morton", [False, True], ids=["random", "morton"])
def test_large_fps_full(morton):
    cfg = inputs.CONFIGS["large"]
    x = inputs.large(morton=morton)
    idx = gpu_fps(x, cfg["npoint"], 0)
    assert_idx_equal(idx, oracle.fps(x, cfg["npoint"], 0), "fps large")


@pytest.mark.slow
@pytest.mark.parametrize("morton", [False, True], ids=["random", "morton"])
def test_large_knn_full(morton):
    """All 100,000 rows of the 100k x 100k kNN against the oracle (the
    spatially ordered kernel with its seed pass), then the row properties."""
    cfg = inputs.CONFIGS["large"]
    x = cache.large(morton)
    k = cfg["knn_k"]
    d, i = gpu_knn(x, x, k)                       # all 100k queries
    wd, wi = cache.large_knn(morton)
    assert_idx_equal(i, wi, "knn large, every row")
    assert_dist_equal(d, wd, "knn large, every row")
    knn_row_properties(x, x, d, i)
    # a point is its own nearest neighbor unless a smaller-index duplicate exists
    assert (d[:, 0] == 0).all()


@pytest.mark.parametrize("morton", [False, True], ids=["random", "morton"])
def test_large_ball_query_full(morton):
    """All 100,000 rows of the Ball Query r=0.02 K=32 against the oracle."""
    cfg = inputs.CONFIGS["large"]
    x = cache.large(morton)
    (r, K), = cfg["bq"]
    d2, i = gpu_bq(x, x, r, K)
    wd2, wi = cache.large_ball_query(morton)
    assert_idx_equal(i, wi, "bq large, every row")
    assert_dist_equal(d2, wd2, "bq large, every row")
    bq_row_properties(x, x, r, d2, i)


# --------------------------------------------------------------------------
# workload 5: 1M points, 1% duplicates; FPS 16384; kNN / BQ of the centers
# --------------------------------------------------------------------------
@pytest.fixture(scope="module")
def very_large():
    x, centers_idx, _ = cache.very_large()         # the oracle's centers
    return inputs.CONFIGS["very_large"], x, centers_idx


@pytest.mark.slow
def test_very_large_fps_full(very_large):
    cfg, x, want = very_large
    idx = gpu_fps(x, cfg["npoint"], 0)
    assert_idx_equal(idx[0], want, "fps very_large")


@pytest.mark.slow
def test_very_large_knn_full(very_large):
    """kNN k=32 of all 16,384 centres against the 1M-point cloud (the ordered
    kernel splits the references into parts), every row against the oracle."""
    cfg, x, cidx = very_large
    q = np.ascontiguousarray(x[:, cidx])
    k = cfg["knn_k"]
    d, i = gpu_knn(q, x, k)
    wd, wi = cache.very_large_knn()
    assert_idx_equal(i, wi, "knn very_large, every row")
    assert_dist_equal(d, wd, "knn very_large, every row")
    knn_row_properties(q, x, d, i)


@pytest.mark.slow
def test_very_large_ball_query_boundary(very_large):
    from _boundary import boundary_points
    cfg, x, cidx = very_large
    (r, K), = cfg["bq"]
    centers = x[0, cidx]
    reject, accept = boundary_points(centers, r, 1500, seed=5)
    assert len(reject) >= 500 and len(accept) >= 500
    # put the boundary points at random non-center positions of the cloud
    ref = x.copy()
    is_center = np.zeros(x.shape[1], bool)
    is_center[cidx] = True
    free = np.nonzero(~is_center)[0]
    rng = np.random.default_rng(6)
    pos = rng.choice(free, size=len(reject) + len(accept), replace=False)
    for p, (_, pt) in zip(pos, reject + accept):
        ref[0, p] = pt
    q = np.ascontiguousarray(x[:, cidx])
    d2, i = gpu_bq(q, ref, r, K)
    bq_row_properties(q, ref, r, d2, i)
    wd2, wi = oracle.ball_query(q, ref, r, K, threads=THREADS)
    assert_idx_equal(i, wi, "bq very_large, every row")
    assert_dist_equal(d2, wd2, "bq very_large, every row")
    # every boundary point is decided the way the contract says
    nrej = nacc = 0
    for p, (c, _) in zip(pos[:len(reject)], reject):
        assert p not in set(i[c].tolist())
        nrej += 1
    for p, (c, _) in zip(pos[len(reject):], accept):
        row = i[c]
        if (row >= 0).sum() < K:
            assert p in set(row.tolist())
            nacc += 1
    assert nrej >= 500 and nacc >= 400


# --------------------------------------------------------------------------
# clouds translated far from the origin: the filter's frame is centred on
# the cloud, but the slack of its bound grows with the squared distance of
# the points from that centre relative to the selection bound, and far from
# the origin coordinates are coarse (spacing 1/1024 at 1e4, 1/32 at 3e5,
# 1/16 at 1e6), so exact ties abound
# --------------------------------------------------------------------------
def translated(x, offset):
    return (x.astype(np.float64) + offset).astype(np.float32)


@pytest.mark.parametrize("offset", [1e4, 3e5, 1e6])
def test_translated_pointnet2_all_kernels(offset):
    """Workload-3 geometry (16 clouds of 4096 points) moved by `offset`:
    FPS, the lane kNN (k=16 of the centres, three_nn k=3), the warp-list kNN
    (k=64) and Ball Query (r=0.1 K=32, r=0.2 K=64), every row against the
    oracle."""
    cfg = inputs.CONFIGS["pointnet2"]
    x = translated(inputs.pointnet2(), offset)
    want = oracle.fps(x, cfg["npoint"], 0, threads=THREADS)
    assert_idx_equal(gpu_fps(x, cfg["npoint"], 0), want, f"fps +{offset:g}")
    c = np.ascontiguousarray(np.take_along_axis(x, want[..., None], axis=1))
    check_knn(c, x, 16, what=f"lane knn +{offset:g}")
    check_knn(x, c, 3, what=f"three_nn +{offset:g}")
    check_knn(c, x, 64, what=f"warp-list knn k=64 +{offset:g}")
    for r, K in cfg["bq"]:
        check_bq(c, x, r, K, what=f"bq +{offset:g} r={r}")


@pytest.mark.parametrize("offset", [1e4, 3e5, -1e6])
def test_translated_ordered_knn_and_ball_query(offset):
    """A 20,000-point mixture cloud moved by `offset`, every point a query:
    the spatially ordered kNN (k=16) and Ball Query (r=0.02 scaled to the
    coordinate spacing), every row against the oracle."""
    rng = np.random.default_rng(int(abs(offset)) % 1000 + 31)
    means = rng.random((16, 3))
    pick = rng.integers(0, 16, 20000)
    x = (means[pick] + rng.standard_normal((20000, 3)) * 0.05)[None]
    x = translated(x.astype(np.float32), offset)
    check_knn(x, x, 16, what=f"ordered knn +{offset:g}")
    r = max(0.02, 4 * float(np.spacing(np.float32(abs(offset)))))
    check_bq(x, x, r, 32, what=f"bq +{offset:g} r={r}")


# --------------------------------------------------------------------------
# edge cases: ragged sizes, misaligned clouds, k / K around warp multiples
# --------------------------------------------------------------------------
@pytest.mark.parametrize("B,Q,N,k", [
    (1, 1, 1, 1), (1, 5, 7, 7), (3, 33, 301, 31), (2, 65, 1001, 33),
    (5, 130, 257, 64), (2, 17, 999, 65), (1, 40, 3000, 128), (2, 9, 700, 256),
    (4, 300, 5, 3),
])
def test_knn_edge_sizes(B, Q, N, k):
    x = inputs.random_cloud(100 + N, B, N, grid=1 / 16)   # many exact ties
    q = inputs.random_cloud(200 + Q, B, Q, grid=1 / 16)
    check_knn(q, x, k, what=f"knn B={B} Q={Q} N={N} k={k}")


@pytest.mark.parametrize("B,Q,N,r,K", [
    (1, 1, 0, 0.5, 4), (2, 7, 0, 0.5, 3), (1, 3, 1, 0.5, 1), (3, 33, 301, 0.4, 31),
    (2, 65, 1001, 0.3, 33), (5, 130, 257, 0.8, 65), (2, 17, 999, 2.5, 16),
    (1, 40, 3000, 0.2, 100), (4, 300, 5, 0.9, 2),
])
def test_ball_query_edge_sizes(B, Q, N, r, K):
    x = inputs.random_cloud(300 + N, B, N, grid=1 / 16)
    q = inputs.random_cloud(400 + Q, B, Q, grid=1 / 16)
    check_bq(q, x, r, K, what=f"bq B={B} Q={Q} N={N} r={r} K={K}")


@pytest.mark.parametrize("B,Q,N", [(1, 100, 2000), (3, 57, 1333)])
def test_random_coordinates_bit_exact(B, Q, N):
    """Non-grid coordinates: every operation rounds, so any difference in the
    arithmetic (contraction, rounding mode, flushing) shows in the distances."""
    x = inputs.random_cloud(500 + N, B, N)
    q = inputs.random_cloud(600 + Q, B, Q)
    check_knn(q, x, 24, what="knn random coordinates")
    check_bq(q, x, 0.45, 48, what="bq random coordinates")
    idx = gpu_fps(x, 200, 1)
    assert_idx_equal(idx, oracle.fps(x, 200, 1), "fps random coordinates")


@pytest.mark.parametrize("B,Q,N,r,K", [
    (1, 64, 100_000, 0.05, 40),     # few hits: every part scans its range
    (2, 300, 70_000, 0.35, 16),     # many hits: the first parts fill K
    (3, 41, 33_000, 0.12, 64),      # ragged tiles and parts
])
def test_ball_query_reference_parts(B, Q, N, r, K):
    """Few queries against many references: the references are split into
    parts whose first-K hits are joined in order; every row against the
    oracle, also with lengths masks."""
    x = inputs.random_cloud(900 + N, B, N)
    q = inputs.random_cloud(901 + Q, B, Q)
    q[:, :5] = x[:, :5]                       # exact matches (distance 0)
    check_bq(q, x, r, K, what=f"bq parts B={B} Q={Q} N={N}")
    ql = np.array([Q, Q - 7, 3][:B], np.int64)
    rl = np.array([N, N // 2 + 11, 200][:B], np.int64)
    d2, i = pc.pc_ball_query(to_dev(q), to_dev(x), r, K, query_lengths=to_dev(ql),
                             ref_lengths=to_dev(rl))
    wd2, wi = oracle.ball_query_masked(q, x, r, K, ql, rl)
    assert_idx_equal(i.cpu().numpy().reshape(-1, K), wi, "bq parts with lengths")
    assert_dist_equal(d2.cpu().numpy().reshape(-1, K), wd2, "bq parts with lengths")


def test_ball_query_large_radius_early_exit():
    x = inputs.random_cloud(5, 2, 20000)
    q = inputs.random_cloud(6, 2, 500)
    check_bq(q, x, 10.0, 64, what="bq everything inside, first 64")


def test_ball_query_nan_reference_rejected():
    x = inputs.random_cloud(7, 1, 600)
    x[0, ::7, 1] = np.nan
    q = inputs.random_cloud(8, 1, 50)
    check_bq(q, x, 0.9, 40, what="bq with NaN references")


def test_subnormal_distances():
    # coordinates ~1e-21: squares are subnormal; flushing them to zero would
    # change both the ordering and the radius decisions
    x = (inputs.random_cloud(9, 1, 700) * np.float32(1e-21)).astype(np.float32)
    q = (inputs.random_cloud(10, 1, 40) * np.float32(1e-21)).astype(np.float32)
    check_knn(q, x, 20, what="knn subnormal")
    check_bq(q, x, 1.2e-21, 30, what="bq subnormal")
    idx = gpu_fps(x, 50, 0)
    assert_idx_equal(idx, oracle.fps(x, 50, 0), "fps subnormal")


def test_outputs_fully_written_over_sentinels():
    x = inputs.random_cloud(11, 2, 513)
    q = inputs.random_cloud(12, 2, 77)
    qd, xd = to_dev(q), to_dev(x)
    od = torch.full((2, 77, 19), 7.5, device=dev())
    oi = torch.full((2, 77, 19), -7, dtype=torch.int64, device=dev())
    pc.pc_knn(qd, xd, 19, out_dist=od, out_idx=oi)
    wd, wi = oracle.knn(q, x, 19)
    assert_idx_equal(oi.cpu().numpy().reshape(-1, 19), wi, "knn sentinels")
    od2 = torch.full((2, 77, 40), 7.5, device=dev())
    oi2 = torch.full((2, 77, 40), -7, dtype=torch.int64, device=dev())
    pc.pc_ball_query(qd, xd, 0.35, 40, out_dist2=od2, out_idx=oi2)
    wd2, wi2 = oracle.ball_query(q, x, 0.35, 40)
    assert_idx_equal(oi2.cpu().numpy().reshape(-1, 40), wi2, "bq sentinels")
    assert_dist_equal(od2.cpu().numpy().reshape(-1, 40), wd2, "bq sentinels")
    of = torch.full((2, 30), -7, dtype=torch.int64, device=dev())
    pc.pc_fps(xd, 30, 5, out=of)
    assert_idx_equal(of.cpu().numpy(), oracle.fps(x, 30, 5), "fps sentinels")


# --------------------------------------------------------------------------
# FPS: every schedule gives the oracle's result
# --------------------------------------------------------------------------
@pytest.mark.parametrize("strategy,cs,bpc", [
    (pc.PC_FPS_BLOCK, 0, 0), (pc.PC_FPS_CLUSTER, 1, 0), (pc.PC_FPS_CLUSTER, 2, 0),
    (pc.PC_FPS_CLUSTER, 4, 0), (pc.PC_FPS_CLUSTER, 8, 0), (pc.PC_FPS_CLUSTER, 3, 0),
    (pc.PC_FPS_GRID, 0, 2), (pc.PC_FPS_GRID, 0, 7), (pc.PC_FPS_GRID, 0, 0),
    # the two-level grid (clusters, then one slot per cluster) and one level
    (pc.PC_FPS_GRID, 4, 8), (pc.PC_FPS_GRID, 8, 0), (pc.PC_FPS_GRID, 16, 0),
    (pc.PC_FPS_GRID, 1, 0), (pc.PC_FPS_GRID, 1, 12),
])
def test_fps_schedules_agree_with_oracle(strategy, cs, bpc):
    x = inputs.random_cloud(13, 2, 5000, grid=1 / 32)
    idx = gpu_fps(x, 300, 17, strategy=strategy, cluster_size=cs,
                  blocks_per_cloud=bpc)
    assert_idx_equal(idx, oracle.fps(x, 300, 17), f"fps schedule {strategy}/{cs}/{bpc}")


@pytest.mark.parametrize("cs", [16, 13])
def test_fps_cluster_on_100k(cs):
    x = inputs.large()
    idx = gpu_fps(x, 600, 3, strategy=pc.PC_FPS_CLUSTER, cluster_size=cs)
    assert_idx_equal(idx, oracle.fps(x, 600, 3), f"fps cluster {cs}")


@pytest.mark.parametrize("cs", [0, 1, 8])
def test_fps_grid_on_100k(cs):
    x = inputs.large()
    idx = gpu_fps(x, 600, 3, strategy=pc.PC_FPS_GRID, cluster_size=cs)
    assert_idx_equal(idx, oracle.fps(x, 600, 3), f"fps grid, cluster size {cs}")


def test_fps_grid_plan_reports_two_levels():
    st, cs, bpc = pc.pc_fps_plan(1, 1_000_000)
    assert st == pc.PC_FPS_GRID and cs in (4, 8, 16) and bpc % cs == 0
    assert pc.pc_fps_plan(1, 1_000_000, pc.PC_FPS_GRID, 1)[1] == 1
    with pytest.raises(pc.PointCloudError):
        pc.pc_fps_plan(1, 1_000_000, pc.PC_FPS_GRID, 8, 12)   # 12 not a multiple of 8


@pytest.mark.parametrize("N,npoint,start", [(1, 4, 0), (5, 9, 2), (7, 7, 6),
                                            (33, 40, 32), (2049, 100, 2048)])
def test_fps_small_and_exhausted(N, npoint, start):
    x = inputs.random_cloud(14 + N, 3, N)
    idx = gpu_fps(x, npoint, start)
    assert_idx_equal(idx, oracle.fps(x, npoint, start), f"fps N={N}")


def test_fps_all_points_identical():
    x = np.ones((2, 300, 3), np.float32)
    idx = gpu_fps(x, 5, 4)
    assert idx.tolist() == [[4, 0, 0, 0, 0]] * 2


def test_fps_workspace_from_caller():
    x = inputs.random_cloud(15, 1, 3000)
    need = pc.binding.lib().pc_fps_workspace_bytes_ex(1, 3000, 50, pc.PC_FPS_GRID, 5)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=dev())
    idx = pc.pc_fps(to_dev(x), 50, 0, strategy=pc.PC_FPS_GRID, blocks_per_cloud=5,
                    workspace=ws).cpu().numpy()
    assert_idx_equal(idx, oracle.fps(x, 50, 0), "fps caller workspace")


# --------------------------------------------------------------------------
# errors reach the caller; bounded waits end without hanging the GPU
# --------------------------------------------------------------------------
def test_invalid_arguments_raise():
    x = to_dev(inputs.random_cloud(16, 1, 10))
    with pytest.raises(pc.PointCloudError) as e:
        pc.pc_knn(x, x, 11)
    assert e.value.status == 1
    with pytest.raises(pc.PointCloudError):
        pc.pc_ball_query(x, x, -1.0, 3)
    with pytest.raises(pc.PointCloudError):
        pc.pc_fps(x, 3, 10)
    with pytest.raises(ValueError):
        pc.pc_knn(x.double(), x.double(), 2)


def test_host_pointer_rejected_by_abi():
    import ctypes
    L = pc.binding.lib()
    host = np.zeros((1, 8, 3), np.float32)
    out = np.zeros((1, 8, 2), np.int64)
    outd = np.zeros((1, 8, 2), np.float32)
    st = L.pc_knn(host.ctypes.data, 1, 8, host.ctypes.data, 8, 2,
                  outd.ctypes.data, out.ctypes.data, None)
    assert st == 1
    assert "not" in L.pc_last_error_message().decode()


def test_fps_grid_wait_timeout_is_reported():
    """Withhold one block's first exchange: every block's bounded wait runs
    out, the kernel returns, the status word says so, and the GPU stays
    usable."""
    x = inputs.random_cloud(17, 1, 4000)
    pc.pc_set_wait_timeout_ns(2_000_000)       # 2 ms
    pc.pc_debug_set_fps_grid_stall(True)
    try:
        idx = pc.pc_fps(to_dev(x), 20, 0, strategy=pc.PC_FPS_GRID,
                        blocks_per_cloud=4).cpu().numpy()
    finally:
        pc.pc_debug_set_fps_grid_stall(False)
        pc.pc_set_wait_timeout_ns(2_000_000_000)
    assert pc.pc_device_status(reset=True) == 4
    assert idx[0, 0] == 0 and (idx[0, 1:] == -1).all()
    # the context is still usable and the next call is correct
    idx = gpu_fps(x, 20, 0, strategy=pc.PC_FPS_GRID, blocks_per_cloud=4)
    assert_idx_equal(idx, oracle.fps(x, 20, 0), "fps after timeout")


def _rows_stopped_or_exact(i, wi, what):
    """Every row is either the oracle's or all -1 (a block that stopped);
    returns the number of stopped rows."""
    i = np.asarray(i).reshape(wi.shape)
    stopped = (i == -1).all(axis=1)
    bad = int((~stopped & (i != wi).any(axis=1)).sum())
    assert bad == 0, f"{what}: {bad} rows neither stopped nor the oracle's"
    return int(stopped.sum())


@pytest.mark.parametrize("case", ["lane", "few_queries", "ordered", "warp_list",
                                  "ball_query", "ball_query_parts"])
def test_tile_stream_wait_timeout_is_reported(case):
    """The producer of the first thread block never issues its first tile's
    copy (nothing is left in flight): its wait and its consumers' run out,
    the kernel returns, the status word says so, the stopped block's rows are
    -1, every other row is the oracle's, and the next call is correct."""
    if case == "ordered":        # spatially ordered kNN: many blocks
        x = cache.large(False)[:, :20000].copy()
        q, k = x, 16
    elif case == "ball_query_parts":   # references split into parts
        x = cache.large(False).copy()
        q, k = np.ascontiguousarray(x[:, :64]), 16
    else:
        # lane: the lane kernel over 32 blocks; few_queries: 64 queries go to
        # the warp-list kernel (8 blocks); warp_list and ball_query: one block
        nq = {"lane": 2000, "few_queries": 64}.get(case, 8)
        x = inputs.random_cloud(30, 1, 3000)
        q = inputs.random_cloud(31, 1, nq)
        k = 40 if case == "warp_list" else 8
    pc.pc_set_wait_timeout_ns(2_000_000)       # 2 ms
    pc.pc_debug_set_stall(pc.PC_STALL_TILE_STREAM)
    try:
        if case.startswith("ball_query"):
            _, got = pc.pc_ball_query(to_dev(q), to_dev(x), 0.5, 16)
        else:
            _, got = pc.pc_knn(to_dev(q), to_dev(x), k)
        got = got.cpu().numpy()
    finally:
        pc.pc_debug_set_stall(0)
        pc.pc_set_wait_timeout_ns(2_000_000_000)
    assert pc.pc_device_status(reset=True) == 4
    if case.startswith("ball_query"):
        _, wi = oracle.ball_query(q, x, 0.5, 16, threads=THREADS)
    else:
        _, wi = oracle.knn(q, x, k, threads=THREADS)
    stopped = _rows_stopped_or_exact(got, wi, case)
    assert stopped >= 1
    if case in ("warp_list", "ball_query"):
        assert stopped == wi.shape[0]          # the only block stopped
    else:
        assert stopped < wi.shape[0]           # only the first block stopped
    # the context is still usable and the next call is correct
    if case.startswith("ball_query"):
        check_bq(q, x, 0.5, 16, what="bq after timeout")
    else:
        check_knn(q, x, k, what=f"{case} knn after timeout")


def test_fps_cluster_wait_timeout_is_reported():
    """Block 0 of the first cloud's cluster withholds its first candidate:
    every block of that cluster runs out its wait, the cloud's remaining
    slots are -1, the other cloud is unaffected, and the next call is
    correct."""
    x = inputs.random_cloud(32, 2, 8000)
    pc.pc_set_wait_timeout_ns(2_000_000)       # 2 ms
    pc.pc_debug_set_stall(pc.PC_STALL_FPS_CLUSTER)
    try:
        idx = pc.pc_fps(to_dev(x), 20, 0, strategy=pc.PC_FPS_CLUSTER,
                        cluster_size=4).cpu().numpy()
    finally:
        pc.pc_debug_set_stall(0)
        pc.pc_set_wait_timeout_ns(2_000_000_000)
    assert pc.pc_device_status(reset=True) == 4
    want = oracle.fps(x, 20, 0)
    assert idx[0, 0] == 0 and (idx[0, 1:] == -1).all()
    assert_idx_equal(idx[1], want[1], "fps cluster, the cloud that did not stall")
    idx = gpu_fps(x, 20, 0, strategy=pc.PC_FPS_CLUSTER, cluster_size=4)
    assert_idx_equal(idx, want, "fps cluster after timeout")


def test_concurrent_streams_equal_serial():
    """FPS, kNN and Ball Query issued on three streams at once (the benchmark
    step) give exactly the results of the same calls one after another."""
    x = to_dev(inputs.large())
    serial = (pc.pc_fps(x, 256, 0), *pc.pc_knn(x, x, 16), *pc.pc_ball_query(x, x, 0.02, 32))
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(main)
    s2.wait_stream(main)
    f = pc.pc_fps(x, 256, 0)
    with torch.cuda.stream(s1):
        kd, ki = pc.pc_knn(x, x, 16)
    with torch.cuda.stream(s2):
        bd, bi = pc.pc_ball_query(x, x, 0.02, 32)
    torch.cuda.synchronize()
    for a, b in zip(serial, (f, kd, ki, bd, bi)):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                           b.view(torch.int32) if b.dtype == torch.float32 else b)
