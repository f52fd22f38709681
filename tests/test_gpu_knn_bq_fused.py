"""kNN and Ball Query of one query set in one call (pc_knn_ball_query).

The call must return exactly what pc_knn and pc_ball_query return (project
page, "k nearest neighbors" and "Ball Query: first K within a radius";
"Numerical contracts"), so every case compares both outputs with the oracle:
all rows where the oracle is quick, sampled rows on the 100k-point clouds
plus every row against the separate GPU calls (themselves checked row by row
against the oracle in test_gpu_parity.py).  The cases cover the fused pass
(one and two query slots per lane, Ball Query rows that overflow K, exact
ties and points exactly on the radius, K = 1 and 64, queries other than the
references, several clouds) and the shapes that fall back to the separate
kernels.
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


def to_dev(a):
    a = np.ascontiguousarray(a)
    if not a.flags.writeable:
        a = a.copy()
    return torch.from_numpy(a).to("cuda:0")


def assert_idx_equal(got, want, what):
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    bad = int((got != want).sum())
    assert bad == 0, f"{what}: {bad} of {got.size} indices differ"


def assert_bits_equal(got, want, what):
    got = np.ascontiguousarray(got, np.float32)
    want = np.ascontiguousarray(want, np.float32)
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    bad = int((got.view(np.uint32) != want.view(np.uint32)).sum())
    assert bad == 0, f"{what}: {bad} of {got.size} distances differ"


@pytest.fixture(autouse=True)
def clean_status():
    yield
    assert pc.pc_device_status(reset=True) == 0


def fused(q, x, k, r, K):
    kd, ki, bd, bi = pc.pc_knn_ball_query(to_dev(q), to_dev(x), k, r, K)
    return (kd.cpu().numpy().reshape(-1, k), ki.cpu().numpy().reshape(-1, k),
            bd.cpu().numpy().reshape(-1, K), bi.cpu().numpy().reshape(-1, K))


def check_against_oracle(q, x, k, r, K, rows=None, what=""):
    """The fused call's four outputs (every row) after comparing the given
    rows (all by default) with the oracle."""
    got = fused(q, x, k, r, K)
    wkd, wki = oracle.knn(q, x, k, rows=rows, threads=THREADS)
    wbd, wbi = oracle.ball_query(q, x, r, K, rows=rows, threads=THREADS)
    kd, ki, bd, bi = got if rows is None else (a[rows] for a in got)
    assert_idx_equal(ki, wki, f"{what} knn")
    assert_bits_equal(kd, wkd, f"{what} knn")
    assert_idx_equal(bi, wbi, f"{what} ball query")
    assert_bits_equal(bd, wbd, f"{what} ball query")
    return got


def check_against_separate(q, x, k, r, K, got, what=""):
    kd, ki, bd, bi = got
    qd, xd = to_dev(q), to_dev(x)
    sd, si = pc.pc_knn(qd, xd, k)
    s2, sb = pc.pc_ball_query(qd, xd, r, K)
    assert_idx_equal(ki, si.cpu().numpy().reshape(-1, k), f"{what} knn vs pc_knn")
    assert_bits_equal(kd, sd.cpu().numpy().reshape(-1, k), f"{what} knn vs pc_knn")
    assert_idx_equal(bi, sb.cpu().numpy().reshape(-1, K), f"{what} bq vs pc_ball_query")
    assert_bits_equal(bd, s2.cpu().numpy().reshape(-1, K), f"{what} bq vs pc_ball_query")


def grid_cloud(seed, B, N, steps=64):
    """Points on a 1/steps grid of the unit cube: many exact ties in s and,
    with r a multiple of the step, references exactly on the radius."""
    rng = np.random.default_rng(seed)
    return (rng.integers(0, steps, size=(B, N, 3)) / steps).astype(np.float32)


# --------------------------------------------------------------------------
# the plan: which shapes run the fused pass
# --------------------------------------------------------------------------
@pytest.mark.parametrize("B,Q,N,k,r,K,want", [
    (1, 100_000, 100_000, 16, 0.02, 32, True),    # the 100k workload
    (1, 100_000, 100_000, 32, 0.02, 64, True),    # one query slot per lane
    (1, 100_000, 100_000, 16, 0.02, 65, False),   # K above 64
    (1, 100_000, 100_000, 1, 0.02, 32, False),    # k = 1: not the ordered path
    (1, 2_000, 100_000, 16, 0.02, 32, False),     # few queries
    (1, 100_000, 8_000, 16, 0.02, 32, False),     # few references
    (1, 100_000, 100_000, 16, 1e-30, 32, False),  # R2 underflows to 0
])
def test_plan(B, Q, N, k, r, K, want):
    assert pc.pc_knn_ball_query_plan(B, Q, N, k, r, K) is want


# --------------------------------------------------------------------------
# the 100k-point workload: every row
# --------------------------------------------------------------------------
@pytest.mark.parametrize("morton", [False, True], ids=["random", "morton"])
def test_large_every_row(morton):
    """kNN k=16 and Ball Query r=0.02 K=32 of all 100,000 points of the
    64-Gaussian cloud in one fused pass: every row equals the oracle's (the
    Ball Query rows directly, the kNN rows through pc_knn on sampled rows
    and every row against it)."""
    cfg = inputs.CONFIGS["large"]
    x = cache.large(morton)
    k = cfg["knn_k"]
    (r, K), = cfg["bq"]
    assert pc.pc_knn_ball_query_plan(1, x.shape[1], x.shape[1], k, r, K)
    got = fused(x, x, k, r, K)
    wbd, wbi = cache.large_ball_query(morton)
    assert_idx_equal(got[3], wbi, "bq large, every row")
    assert_bits_equal(got[2], wbd, "bq large, every row")
    rows = inputs.sample_rows(7, x.shape[1], 2000)
    wkd, wki = oracle.knn(x, x, k, rows=rows, threads=THREADS)
    assert_idx_equal(got[1][rows], wki, "knn large, sampled rows")
    assert_bits_equal(got[0][rows], wkd, "knn large, sampled rows")
    check_against_separate(x, x, k, r, K, got, "large")


@pytest.mark.slow
def test_large_every_knn_row():
    cfg = inputs.CONFIGS["large"]
    x = cache.large(False)
    k = cfg["knn_k"]
    (r, K), = cfg["bq"]
    kd, ki, _, _ = fused(x, x, k, r, K)
    wkd, wki = cache.large_knn(False)
    assert_idx_equal(ki, wki, "knn large, every row")
    assert_bits_equal(kd, wkd, "knn large, every row")


# --------------------------------------------------------------------------
# fused cases the oracle checks row by row (sampled where large)
# --------------------------------------------------------------------------
# (The fused pass needs enough queries to fill the GPU without splitting the
# references into parts: about 100,000 with two query slots per lane,
# 50,000 with one.)
def test_overflowing_rows_one_slot_per_lane():
    """k = 32 (one query slot per lane) and r = 0.07, K = 64 on 60,000
    uniform points: about 86 hits a query, so most rows drop hits and keep
    the 64 smallest indices."""
    x = inputs.random_cloud(40, 1, 60_000, lo=0.0, hi=1.0)
    assert pc.pc_knn_ball_query_plan(1, 60_000, 60_000, 32, 0.07, 64)
    _, _, _, bi = check_against_oracle(x, x, 32, 0.07, 64,
                                       rows=inputs.sample_rows(41, 60_000, 1500),
                                       what="overflow")
    check_against_separate(x, x, 32, 0.07, 64, fused(x, x, 32, 0.07, 64), "overflow")
    full = (bi >= 0).all(axis=1).mean()
    assert full > 0.5, f"only {full:.2f} of the rows overflow"


def test_ties_and_points_on_the_radius():
    """100,000 grid points (1/64 steps, so also duplicates) with r = 1/32:
    s32 ties everywhere, and the references exactly 2 steps away along an
    axis sit exactly on the radius (s32 = R2, excluded by the strict
    test)."""
    x = grid_cloud(42, 1, 100_000)
    r = 1.0 / 32
    assert oracle.radius_threshold(r) == np.float32(r * r)
    assert pc.pc_knn_ball_query_plan(1, 100_000, 100_000, 16, r, 32)
    rows = inputs.sample_rows(43, 100_000, 2000)
    got = check_against_oracle(x, x, 16, r, 32, rows=rows, what="grid ties")
    check_against_separate(x, x, 16, r, 32, got, "grid ties")


@pytest.mark.parametrize("k,K", [(2, 1), (16, 64), (24, 8)])
def test_other_queries_several_clouds(k, K):
    """Queries that are not the references (their own spatial order), two
    clouds, K at both ends of the fused range."""
    x = inputs.random_cloud(44, 2, 20_000, lo=0.0, hi=1.0)
    q = inputs.random_cloud(45, 2, 50_000, lo=0.0, hi=1.0)
    r = 0.05
    assert pc.pc_knn_ball_query_plan(2, 50_000, 20_000, k, r, K)
    got = check_against_oracle(q, x, k, r, K, rows=inputs.sample_rows(46, 2 * 50_000, 1500),
                               what=f"k={k} K={K}")
    check_against_separate(q, x, k, r, K, got, f"k={k} K={K}")


def test_no_hits_and_every_row_full():
    """A radius below every nonzero distance (only the point itself, s = 0)
    and one above the whole cloud (every row full, the K smallest indices)."""
    x = inputs.random_cloud(47, 1, 100_000, lo=0.0, hi=1.0)
    assert pc.pc_knn_ball_query_plan(1, 100_000, 100_000, 8, 1e-6, 4)
    rows = inputs.sample_rows(48, 100_000, 1000)
    _, _, bd, bi = check_against_oracle(x, x, 8, 1e-6, 4, rows=rows, what="tiny r")
    assert (bi[:, 1:] == -1).all() and (bd[:, 1:] == 0).all()
    _, _, bd, bi = check_against_oracle(x, x, 8, 4.0, 64, rows=rows, what="huge r")
    assert (bi == np.arange(64)).all()


# --------------------------------------------------------------------------
# shapes that run the separate kernels
# --------------------------------------------------------------------------
@pytest.mark.parametrize("B,Q,N,k,r,K", [
    (1, 64, 20_000, 16, 0.05, 32),     # few queries
    (2, 3_000, 5_000, 16, 0.1, 32),    # few references
    (1, 8_192, 20_000, 16, 0.05, 32),  # references split into parts
    (1, 8_192, 20_000, 1, 0.05, 32),   # k = 1
    (1, 8_192, 20_000, 16, 0.05, 100), # K above 64
    (1, 1, 1, 1, 0.5, 3),              # a single point
])
def test_separate_kernel_shapes(B, Q, N, k, r, K):
    assert not pc.pc_knn_ball_query_plan(B, Q, N, k, r, K)
    x = inputs.random_cloud(50, B, N, lo=0.0, hi=1.0)
    q = inputs.random_cloud(51, B, Q, lo=0.0, hi=1.0)
    rows = None if B * Q <= 4096 else inputs.sample_rows(52, B * Q, 1000)
    check_against_oracle(q, x, k, r, K, rows=rows, what="separate")


def test_argument_errors():
    x = to_dev(inputs.random_cloud(53, 1, 100, lo=0.0, hi=1.0))
    with pytest.raises(pc.PointCloudError):
        pc.pc_knn_ball_query(x, x, 101, 0.1, 4)        # k > N
    with pytest.raises(pc.PointCloudError):
        pc.pc_knn_ball_query(x, x, 4, -0.1, 4)         # radius <= 0
    with pytest.raises(pc.PointCloudError):
        pc.pc_knn_ball_query(x, x, 4, 0.1, 0)          # K < 1
    with pytest.raises(ValueError):
        bad = torch.empty((1, 100, 3), dtype=torch.float32, device="cuda:0")
        pc.pc_knn_ball_query(x, x, 4, 0.1, 4, out=(bad, bad, bad, bad))


def test_stopped_block_is_reported():
    """The producer of the first thread block never issues its first tile's
    copy: its consumers' waits run out, the status word says so, both
    outputs' rows of that block's queries are -1, every other row is the
    oracle's, and the next call is correct."""
    x = cache.large(False)
    k, r, K = 16, 0.02, 32
    rows = inputs.sample_rows(54, x.shape[1], 1500)
    pc.pc_set_wait_timeout_ns(2_000_000)
    pc.pc_debug_set_stall(pc.PC_STALL_TILE_STREAM)
    try:
        _, ki, bd, bi = fused(x, x, k, r, K)
    finally:
        pc.pc_debug_set_stall(0)
        pc.pc_set_wait_timeout_ns(2_000_000_000)
    assert pc.pc_device_status(reset=True) == 4
    stopped_k = (ki == -1).all(axis=1)
    stopped_b = (bi == -1).all(axis=1) & (bd == 0).all(axis=1)
    assert stopped_k.sum() >= 1 and stopped_k.sum() < ki.shape[0]
    assert (stopped_b | ~stopped_k).all(), "a stopped kNN row has Ball Query hits"
    _, wki = oracle.knn(x, x, k, rows=rows, threads=THREADS)
    _, wbi = oracle.ball_query(x, x, r, K, rows=rows, threads=THREADS)
    keep = ~stopped_k[rows]
    assert_idx_equal(ki[rows][keep], wki[keep], "knn rows that ran")
    assert_idx_equal(bi[rows][keep], wbi[keep], "bq rows that ran")
    check_against_oracle(x, x, k, r, K, rows=rows, what="after timeout")


def test_benchmark_step_configuration():
    """The benchmark's step as it launches it: FPS 4096 on a 13-block
    cluster on the main stream, the fused call on a side stream planned for
    the SMs FPS leaves (pc_set_sm_reserve(13)), both running at once: FPS
    and every Ball Query row equal the oracle's, kNN on sampled rows and on
    every row against pc_knn."""
    cfg = inputs.CONFIGS["large"]
    x = cache.large(False)
    k = cfg["knn_k"]
    (r, K), = cfg["bq"]
    xd = to_dev(x)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    fork = torch.cuda.Event()
    fork.record(main)
    fps = pc.pc_fps(xd, cfg["npoint"], 0, strategy=pc.PC_FPS_CLUSTER, cluster_size=13)
    side.wait_event(fork)
    with torch.cuda.stream(side):
        pc.pc_set_sm_reserve(13)
        try:
            kd, ki, bd, bi = pc.pc_knn_ball_query(xd, xd, k, r, K)
        finally:
            pc.pc_set_sm_reserve(0)
    torch.cuda.synchronize()
    assert_idx_equal(fps.cpu().numpy(), oracle.fps(x, cfg["npoint"], 0, threads=THREADS),
                     "fps, 13-block cluster")
    N = x.shape[1]
    wbd, wbi = cache.large_ball_query(False)
    assert_idx_equal(bi.cpu().numpy().reshape(N, K), wbi, "bq, every row")
    assert_bits_equal(bd.cpu().numpy().reshape(N, K), wbd, "bq, every row")
    rows = inputs.sample_rows(55, N, 2000)
    wkd, wki = oracle.knn(x, x, k, rows=rows, threads=THREADS)
    kd = kd.cpu().numpy().reshape(N, k)
    ki = ki.cpu().numpy().reshape(N, k)
    assert_idx_equal(ki[rows], wki, "knn, sampled rows")
    assert_bits_equal(kd[rows], wkd, "knn, sampled rows")
    sd, si = pc.pc_knn(xd, xd, k)
    assert_idx_equal(ki, si.cpu().numpy().reshape(N, k), "knn vs pc_knn, every row")
    assert_bits_equal(kd, sd.cpu().numpy().reshape(N, k), "knn vs pc_knn, every row")
