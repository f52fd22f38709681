"""FPS of the BLOCK and CLUSTER schedules against the oracle on the cases
where a per-block reduction or the exchange between blocks could go wrong.
The CLUSTER cases run both kernels: the rounds kernel (default; several
centers certified per exchange) and one center per exchange
(pc_fps_set_batched(False)).

The operator (mps-pointops project page, "Farthest point sampling";
"Contracts"): c_0 = start; each step takes the point with the largest
minimum squared distance to the centers so far, the smallest index on an
exact tie.  Cases: exact ties between points of different blocks
(coordinates on a grid, duplicates) for every cluster size up to 16,
clouds exhausted to m = 0 everywhere, coarse coordinates far from the
origin, the 100k-point cloud on the benchmark step's 13-block cluster in
both storage orders, and many clouds on the BLOCK schedule.
"""
import numpy as np
import pytest
import torch

import oracle
import point_cloud_neighbor_gb300 as pc
from point_cloud_neighbor_gb300 import inputs

pytestmark = pytest.mark.gpu

THREADS = oracle.default_threads()


@pytest.fixture(params=[True, False], ids=["rounds", "per_step"])
def batched(request):
    prev = pc.pc_fps_set_batched(request.param)
    yield request.param
    pc.pc_fps_set_batched(prev)


@pytest.fixture(autouse=True)
def clean_status():
    yield
    assert pc.pc_device_status(reset=True) == 0


def gpu_fps(x, npoint, start=0, **kw):
    xd = torch.from_numpy(np.ascontiguousarray(x)).to("cuda:0")
    return pc.pc_fps(xd, npoint, start, **kw).cpu().numpy()


def assert_idx_equal(got, want, what):
    assert got.shape == want.shape, f"{what}: shape {got.shape} vs {want.shape}"
    bad = int((got != want).sum())
    assert bad == 0, f"{what}: {bad} of {got.size} indices differ"


@pytest.mark.parametrize("strategy,cs", [
    (pc.PC_FPS_BLOCK, 0), (pc.PC_FPS_CLUSTER, 1), (pc.PC_FPS_CLUSTER, 2),
    (pc.PC_FPS_CLUSTER, 3), (pc.PC_FPS_CLUSTER, 8), (pc.PC_FPS_CLUSTER, 13),
    (pc.PC_FPS_CLUSTER, 16),
])
def test_grid_ties_every_cluster_size(batched, strategy, cs):
    """Two clouds of 6,000 points on a 1/32 grid (duplicates and equal
    distances everywhere), 700 samples from start 11."""
    x = inputs.random_cloud(60, 2, 6000, grid=1 / 32)
    want = oracle.fps(x, 700, 11, threads=THREADS)
    got = gpu_fps(x, 700, 11, strategy=strategy, cluster_size=cs)
    assert_idx_equal(got, want, f"grid ties {strategy}/{cs}")


def test_exhausted_cloud(batched):
    """8,192 points at 40 distinct places (each repeated): after 40 samples
    every minimum is 0 and the rest repeat the smallest index, 0."""
    rng = np.random.default_rng(61)
    places = rng.random((40, 3)).astype(np.float32)
    x = places[rng.integers(0, 40, size=(1, 8192))]
    want = oracle.fps(x, 120, 5, threads=THREADS)
    got = gpu_fps(x, 120, 5, strategy=pc.PC_FPS_CLUSTER, cluster_size=4)
    assert_idx_equal(got, want, "exhausted")
    assert (got[0, 40:] == 0).all()


@pytest.mark.parametrize("offset", [1e4, 1e6])
def test_far_from_the_origin(batched, offset):
    """Coordinates of 1e4 and 1e6 (spacing 1/1024 and 1/16): few distinct
    distances, many exact ties, boxes whose bound is often exactly tight."""
    x = (inputs.random_cloud(62, 2, 12_000, lo=0.0, hi=64.0).astype(np.float64) +
         offset).astype(np.float32)
    want = oracle.fps(x, 900, 0, threads=THREADS)
    got = gpu_fps(x, 900, 0)
    assert_idx_equal(got, want, f"offset {offset:g}")


@pytest.mark.parametrize("morton", [False, True], ids=["random", "morton"])
def test_large_cloud_step_schedule(batched, morton):
    """The 100k-point cloud, 4,096 samples, on a cluster of 13 blocks (the
    schedule of the benchmark step)."""
    x = inputs.large(morton=morton)
    want = oracle.fps(x, 4096, 0, threads=THREADS)
    got = gpu_fps(x, 4096, 0, strategy=pc.PC_FPS_CLUSTER, cluster_size=13)
    assert_idx_equal(got, want, "large, cluster 13")


def test_many_clouds_block_schedule():
    """96 clouds of 4,096 points (one block each: the BLOCK schedule)."""
    x = inputs.random_cloud(63, 96, 4096)
    want = oracle.fps(x, 256, 3, threads=THREADS)
    got = gpu_fps(x, 256, 3, strategy=pc.PC_FPS_BLOCK)
    assert_idx_equal(got, want, "96 clouds")


def test_switch_returns_previous():
    prev = pc.pc_fps_set_batched(False)
    try:
        assert pc.pc_fps_set_batched(True) is False
        assert pc.pc_fps_set_batched(True) is True
    finally:
        pc.pc_fps_set_batched(prev)


def test_cluster_wait_timeout(batched):
    """Block 0 of the first cloud withholds its first candidates (its first
    round's list): that cloud's slots after the start are -1, the other
    cloud is exact, the status word says PC_ERR_DEVICE_TIMEOUT, and the next
    call is correct."""
    x = inputs.random_cloud(64, 2, 8000)
    pc.pc_set_wait_timeout_ns(2_000_000)
    pc.pc_debug_set_stall(pc.PC_STALL_FPS_CLUSTER)
    try:
        idx = gpu_fps(x, 20, 0, strategy=pc.PC_FPS_CLUSTER, cluster_size=4)
    finally:
        pc.pc_debug_set_stall(0)
        pc.pc_set_wait_timeout_ns(2_000_000_000)
    assert pc.pc_device_status(reset=True) == 4
    want = oracle.fps(x, 20, 0)
    assert idx[0, 0] == 0 and (idx[0, 1:] == -1).all()
    assert_idx_equal(idx[1], want[1], "the cloud that did not stall")
    assert_idx_equal(gpu_fps(x, 20, 0, strategy=pc.PC_FPS_CLUSTER, cluster_size=4), want,
                     "after the timeout")


@pytest.mark.parametrize("npoint", [1, 2, 65, 300])
def test_short_runs(batched, npoint):
    """Few samples (a run cut by npoint), 3 clouds on clusters of 8."""
    x = inputs.random_cloud(65, 3, 9000)
    assert_idx_equal(gpu_fps(x, npoint, 7, strategy=pc.PC_FPS_CLUSTER, cluster_size=8),
                     oracle.fps(x, npoint, 7), f"npoint={npoint}")


@pytest.fixture(scope="module")
def large_fps_oracle():
    """The oracle's 4096 samples of the 100k-point cloud and of its first
    90,000 points (computed once)."""
    out = {}
    for name, x in (("100k", inputs.large()), ("90k", inputs.large()[:, :90000].copy())):
        out[name] = (x, oracle.fps(x, 4096, 0, threads=THREADS))
    return out


@pytest.mark.parametrize("cloud", ["100k", "90k"])
@pytest.mark.parametrize("cs", [11, 12, 13, 14, 15, 16])
def test_rounds_every_cluster_size_large(large_fps_oracle, cloud, cs):
    """Every block of a cloud must certify the same run from the same lists:
    with more candidates above the bound than a run can hold, the ones kept
    must not depend on the warps' timing (the 100k cloud on 12 blocks and
    the 90k cloud on 16 exceed the candidate capacity in some rounds)."""
    x, want = large_fps_oracle[cloud]
    got = gpu_fps(x, 4096, 0, strategy=pc.PC_FPS_CLUSTER, cluster_size=cs)
    assert_idx_equal(got, want, f"{cloud} on {cs} blocks")


# ---------------------------------------------------------------------------
# The two-level GRID schedule: in rounds, each cluster's leader summarizes
# its blocks' lists and every block certifies the run from all clusters'
# summaries; per step, one slot per cluster.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cs,bpc", [(2, 4), (4, 8), (4, 12), (8, 16), (8, 40), (16, 32)])
def test_grid_two_levels_ties(batched, cs, bpc):
    """Two clouds of 12,000 points on a 1/32 grid (exact ties between points
    of different clusters), 900 samples from start 7."""
    x = inputs.random_cloud(66, 2, 12_000, grid=1 / 32)
    want = oracle.fps(x, 900, 7, threads=THREADS)
    got = gpu_fps(x, 900, 7, strategy=pc.PC_FPS_GRID, cluster_size=cs, blocks_per_cloud=bpc)
    assert_idx_equal(got, want, f"grid ties, {bpc // cs} clusters of {cs}")


def test_grid_two_levels_exhausted(batched):
    """8,192 points at 40 places on 3 clusters of 4: every minimum reaches 0,
    then the slots repeat index 0."""
    rng = np.random.default_rng(67)
    places = rng.random((40, 3)).astype(np.float32)
    x = places[rng.integers(0, 40, size=(1, 8192))]
    want = oracle.fps(x, 120, 5, threads=THREADS)
    got = gpu_fps(x, 120, 5, strategy=pc.PC_FPS_GRID, cluster_size=4, blocks_per_cloud=12)
    assert_idx_equal(got, want, "grid exhausted")


@pytest.mark.parametrize("cloud", ["100k", "90k"])
@pytest.mark.parametrize("cs,bpc", [(16, 32), (16, 48), (8, 40), (4, 36)])
def test_grid_rounds_large(large_fps_oracle, cloud, cs, bpc):
    """The 100k-point cloud and its first 90,000 points, 4096 samples, on
    two-level grids of 2 to 9 clusters: summaries that overflow their 128
    places in some rounds must still give every block the same run."""
    x, want = large_fps_oracle[cloud]
    got = gpu_fps(x, 4096, 0, strategy=pc.PC_FPS_GRID, cluster_size=cs, blocks_per_cloud=bpc)
    assert_idx_equal(got, want, f"{cloud} on {bpc // cs} clusters of {cs}")


def test_grid_rounds_wait_timeout(batched):
    """Cluster 0 of the first cloud withholds its first summary (rounds) or
    its first slot (per step): every bounded wait of that cloud's blocks runs
    out, its slots after the start are -1, the other cloud is exact, the
    status word says so, and the next call is correct."""
    x = inputs.random_cloud(68, 2, 9000)
    pc.pc_set_wait_timeout_ns(2_000_000)
    pc.pc_debug_set_stall(pc.PC_STALL_FPS_GRID)
    try:
        idx = gpu_fps(x, 30, 0, strategy=pc.PC_FPS_GRID, cluster_size=4, blocks_per_cloud=8)
    finally:
        pc.pc_debug_set_stall(0)
        pc.pc_set_wait_timeout_ns(2_000_000_000)
    assert pc.pc_device_status(reset=True) == 4
    assert idx[0, 0] == 0 and (idx[0, 1:] == -1).all()
    want = oracle.fps(x, 30, 0)
    assert_idx_equal(idx[1], want[1], "the cloud that did not stall")
    assert_idx_equal(gpu_fps(x, 30, 0, strategy=pc.PC_FPS_GRID, cluster_size=4,
                             blocks_per_cloud=8), want, "after the timeout")
