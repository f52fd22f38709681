"""GPU parity of the operators built on the hot path: lengths-masked kNN and
Ball Query, Chamfer distance (forward), three_interpolate (forward and
backward), the neighbor gather and the PyTorch3D-style Ball Query adapter.

Indices are compared bit for bit with the oracle, distances and the
three_interpolate forward bit for bit (same operation order); the Chamfer
loss (float64 sums in a different order, one rounding to float32) within one
float32 ulp; the three_interpolate backward bit for bit for M <= 16384
(ordered sums; M <= 16384, n <= 8192), otherwise (atomic adds in any order)
within the bound
2 (s + 1) u sum|w g| per element, s the number of terms.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import point_cloud_neighbor_gb300 as pc
from point_cloud_neighbor_gb300 import inputs
from point_cloud_neighbor_gb300.pytorch3d import ball_query as p3d_ball_query
from test_gpu_parity import THREADS, assert_dist_equal, assert_idx_equal, to_dev

pytestmark = pytest.mark.gpu
U = 2.0 ** -24
GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "quickstart_propagation.json")


@pytest.fixture(autouse=True)
def clean_status():
    yield
    assert pc.pc_device_status(reset=True) == 0


def lens(v):
    return torch.tensor(v, dtype=torch.int64, device="cuda")


def host(t):
    return t.cpu().numpy()


# --- lengths-masked kNN / Ball Query ------------------------------------------
@pytest.mark.parametrize("B,Q,N,k,ql,rl", [
    (3, 40, 300, 5, [40, 17, 0], [300, 4, 299]),
    (2, 257, 513, 33, [1, 257], [513, 256]),
    (4, 70, 100, 64, None, [100, 1, 63, 64]),
    (2, 9, 700, 256, [9, 3], None),
    (1, 31, 12, 16, None, [12]),          # k > N: padded slots
    (2, 5, 0, 3, None, [0, 0]),           # no references at all
])
@pytest.mark.parametrize("squared", [False, True])
def test_knn_ex_lengths_and_squared(B, Q, N, k, ql, rl, squared):
    q = inputs.random_cloud(100 + Q, B, Q, grid=1 / 16)
    x = inputs.random_cloud(200 + N, B, N, grid=1 / 16)
    d, i = pc.pc_knn(to_dev(q), to_dev(x), k,
                     query_lengths=None if ql is None else lens(ql),
                     ref_lengths=None if rl is None else lens(rl), squared=squared)
    wd, wi = oracle.knn_masked(q, x, k, ql, rl, squared=squared, threads=THREADS)
    assert_idx_equal(host(i).reshape(-1, k), wi, "knn_ex")
    assert_dist_equal(host(d).reshape(-1, k), wd, "knn_ex")


def test_knn_ex_lengths_out_of_range_are_clamped():
    q = inputs.random_cloud(1, 2, 20)
    x = inputs.random_cloud(2, 2, 50)
    d, i = pc.pc_knn(to_dev(q), to_dev(x), 4, query_lengths=lens([-3, 99]),
                     ref_lengths=lens([1000, -1]))
    wd, wi = oracle.knn_masked(q, x, 4, [-3, 99], [1000, -1])
    assert_idx_equal(host(i).reshape(-1, 4), wi, "knn_ex clamp")


@pytest.mark.parametrize("B,Q,N,r,K,ql,rl", [
    (3, 40, 300, 0.25, 7, [40, 17, 0], [300, 4, 299]),
    (2, 130, 1000, 0.5, 40, [130, 1], [513, 1000]),
    (2, 33, 257, 5.0, 300, None, [257, 0]),
])
def test_ball_query_ex_lengths(B, Q, N, r, K, ql, rl):
    q = inputs.random_cloud(300 + Q, B, Q, grid=1 / 16)
    x = inputs.random_cloud(400 + N, B, N, grid=1 / 16)
    d2, i = pc.pc_ball_query(to_dev(q), to_dev(x), r, K,
                             query_lengths=None if ql is None else lens(ql),
                             ref_lengths=None if rl is None else lens(rl))
    wd, wi = oracle.ball_query_masked(q, x, r, K, ql, rl)
    assert_idx_equal(host(i).reshape(-1, K), wi, "ball_query_ex")
    assert_dist_equal(host(d2).reshape(-1, K), wd, "ball_query_ex")


# --- Chamfer ------------------------------------------------------------------
def ulp_close(got, want):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    tol = np.spacing(np.maximum(np.abs(got), np.abs(want)).astype(np.float32))
    return bool((np.abs(got.astype(np.float64) - want.astype(np.float64)) <= tol).all())


def check_chamfer(x, y, what, **kw):
    t = {k: (to_dev(np.asarray(v, np.int64)) if k.endswith("lengths") and v is not None
             else to_dev(np.asarray(v, np.float32)) if k == "weights" and v is not None
             else v) for k, v in kw.items()}
    loss, (dx, ix), other = pc.pc_chamfer(to_dev(x), to_dev(y), **t)
    wl, (wdx, wix), wother = oracle.chamfer(x, y, threads=THREADS, **kw)
    assert_idx_equal(host(ix), wix, what + " idx_x")
    assert_dist_equal(host(dx), wdx, what + " dist_x")
    if wother is not None:
        assert_idx_equal(host(other[1]), wother[1], what + " idx_y")
        assert_dist_equal(host(other[0]), wother[0], what + " dist_y")
    assert ulp_close(host(loss), wl), f"{what}: loss {host(loss)} vs {wl}"


def test_chamfer_quickstart():
    g = json.load(open(GOLDEN))
    xyz = np.array(g["xyz"], np.float32)
    loss, _ = pc.chamfer_distance(to_dev(xyz[:, :2]), to_dev(xyz))
    assert float(loss) == np.float32(g["chamfer"]["loss"])


@pytest.mark.parametrize("point_reduction", ["sum", "mean"])
@pytest.mark.parametrize("batch_reduction", ["none", "sum", "mean"])
def test_chamfer_reductions(point_reduction, batch_reduction):
    x = inputs.random_cloud(30, 3, 500)
    y = inputs.random_cloud(31, 3, 333)
    check_chamfer(x, y, f"chamfer {point_reduction}/{batch_reduction}",
                  point_reduction=point_reduction, batch_reduction=batch_reduction)


def test_chamfer_lengths_weights_single_direction():
    x = inputs.random_cloud(32, 4, 300, grid=1 / 32)
    y = inputs.random_cloud(33, 4, 257, grid=1 / 32)
    kw = dict(x_lengths=[300, 1, 0, 150], y_lengths=[257, 100, 5, 0],
              weights=[1.0, 0.5, 2.0, 0.25])
    check_chamfer(x, y, "chamfer lengths+weights", **kw)
    check_chamfer(x, y, "chamfer lengths none", batch_reduction="none", **kw)
    check_chamfer(x, y, "chamfer single", single_directional=True, **kw)


def test_chamfer_point_mae_shape():
    # the pages' Chamfer timing shape: batch 4, up to 16,384 points per cloud;
    # full comparison at 4096 points (the oracle finishes in seconds)
    x = inputs.random_cloud(34, 4, 4096)
    y = inputs.random_cloud(35, 4, 4096)
    check_chamfer(x, y, "chamfer 4x4096")


def test_chamfer_empty():
    x = inputs.random_cloud(36, 2, 10)
    y = np.zeros((2, 0, 3), np.float32)
    check_chamfer(x, y, "chamfer empty y")
    loss, _, _ = pc.pc_chamfer(to_dev(np.zeros((0, 5, 3), np.float32)),
                               to_dev(np.zeros((0, 4, 3), np.float32)))
    assert float(loss) == 0.0


# --- three_interpolate --------------------------------------------------------
def interp_case(seed, B, C, M, n, pad=False):
    rng = np.random.default_rng(seed)
    f = rng.standard_normal((B, C, M)).astype(np.float32)
    idx = rng.integers(0, M, (B, n, 3)).astype(np.int64)
    if pad:
        idx[rng.random((B, n, 3)) < 0.1] = -1
    w = rng.random((B, n, 3)).astype(np.float32)
    return f, idx, w


def test_three_interpolate_quickstart():
    g = json.load(open(GOLDEN))
    xyz = to_dev(np.array(g["xyz"], np.float32))
    d, i = pc.three_nn(xyz[:, :2].contiguous(), xyz)
    assert host(i).tolist() == g["three_nn"]["idx"]
    w = torch.full_like(d, 1.0 / 3.0)
    f = torch.ones((1, 2, 3), device="cuda", requires_grad=True)
    out = pc.three_interpolate(f, i, w)
    assert host(out.detach()).tolist() == g["three_interpolate"]["out"]
    out.sum().backward()
    # each feature column m receives the weights of the slots pointing at it
    want = oracle.three_interpolate_backward(np.ones((1, 2, 2), np.float32),
                                             host(i), host(w), 3)
    assert np.array_equal(host(f.grad), want)


@pytest.mark.parametrize("B,C,M,n,pad", [
    (1, 1, 3, 1, False), (2, 5, 11, 17, True), (3, 33, 100, 130, False),
    (16, 64, 1024, 4096, False), (2, 16, 7, 1000, True),
    (1, 3, 20000, 500, True),   # M above the shared-memory tile: direct kernel
    (2, 40, 16384, 300, False),  # largest staged tile, one channel per block
])
def test_three_interpolate_forward_bit_exact(B, C, M, n, pad):
    f, idx, w = interp_case(40 + n, B, C, M, n, pad)
    out = pc.pc_three_interpolate(to_dev(f), to_dev(idx), to_dev(w))
    want = oracle.three_interpolate(f, idx, w)
    assert np.array_equal(host(out).view(np.int32), want.view(np.int32))


@pytest.mark.parametrize("B,C,M,n,pad", [
    (2, 5, 11, 17, True), (3, 33, 100, 130, False), (16, 32, 1024, 4096, False),
    (1, 3, 2, 2000, False),   # heavy collisions: 3000 terms per element
    (1, 3, 20000, 500, True),  # M above the shared-memory tile: direct kernel
    (2, 5, 300, 0, False),     # no points: the gradient is zero
    (1, 6, 500, 8192, True),   # largest staged grad_out rows
    (1, 2, 64, 9000, False),   # n above the staged rows: atomic kernel
])
def test_three_interpolate_backward_within_bound(B, C, M, n, pad):
    f, idx, w = interp_case(50 + n, B, C, M, n, pad)
    g = np.random.default_rng(60 + n).standard_normal((B, C, n)).astype(np.float32)
    got = host(pc.pc_three_interpolate_backward(to_dev(g), to_dev(idx), to_dev(w), M))
    want = oracle.three_interpolate_backward(g, idx, w, M)
    mag = np.zeros((B, C, M))
    cnt = np.zeros((B, M))
    for b in range(B):
        valid = idx[b] >= 0
        terms = np.abs(w[b][None, :, :].astype(np.float64) *
                       g[b][:, :, None].astype(np.float64))       # [C, n, 3]
        for c in range(C):
            np.add.at(mag[b, c], idx[b][valid], terms[c][valid])
        np.add.at(cnt[b], idx[b][valid], 1)
    if M <= 16384 and n <= 8192:
        # deterministic path: the same summation order as the oracle
        assert np.array_equal(got.view(np.int32), want.view(np.int32))
    bound = 2 * (cnt[:, None, :] + 1) * U * mag + 1e-44
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    assert (err <= bound).all(), f"max excess {(err - bound).max()}"


def test_three_interpolate_bad_index_sets_status():
    f, idx, w = interp_case(70, 1, 2, 5, 4)
    idx[0, 1, 2] = 5
    out = pc.pc_three_interpolate(to_dev(f), to_dev(idx), to_dev(w))
    assert pc.pc_device_status(reset=True) == pc.binding.PC_ERR_INVALID_ARGUMENT
    idx_ok = idx.copy()
    idx_ok[0, 1, 2] = -1
    assert np.array_equal(host(out), oracle.three_interpolate(f, idx_ok, w))


# --- gather and the PyTorch3D-style adapter ------------------------------------
def test_gather_points_matches_oracle():
    x = inputs.random_cloud(80, 3, 50)
    idx = np.random.default_rng(81).integers(-1, 50, (3, 20, 7)).astype(np.int64)
    got = pc.pc_gather_points(to_dev(x), to_dev(idx))
    assert np.array_equal(host(got), oracle.gather_points(x, idx))


def test_pytorch3d_adapter_defaults_and_lengths():
    x = inputs.pointnet2()[:4]
    c = np.ascontiguousarray(x[:, :512])
    res = p3d_ball_query(to_dev(c), to_dev(x))          # K=500, radius=0.2
    wd, wi = oracle.ball_query_masked(c, x, 0.2, 500)
    assert_idx_equal(host(res.idx).reshape(-1, 500), wi, "p3d idx")
    assert_dist_equal(host(res.dists).reshape(-1, 500), wd, "p3d dists")
    assert np.array_equal(host(res.knn), oracle.gather_points(x, wi.reshape(4, 512, 500)))
    l1, l2 = lens([512, 100, 0, 7]), lens([4096, 4096, 10, 0])
    res = p3d_ball_query(to_dev(c), to_dev(x), lengths1=l1, lengths2=l2, K=32,
                         radius=0.1, return_nn=False, skip_points_outside_cube=True)
    assert res.knn is None
    wd, wi = oracle.ball_query_masked(c, x, 0.1, 32, [512, 100, 0, 7],
                                      [4096, 4096, 10, 0])
    assert_idx_equal(host(res.idx).reshape(-1, 32), wi, "p3d lengths")
    assert_dist_equal(host(res.dists).reshape(-1, 32), wd, "p3d lengths")
