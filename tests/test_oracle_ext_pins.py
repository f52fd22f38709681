"""Pins of the oracle's lengths-masked kNN / Ball Query, gather,
three_interpolate and Chamfer (CPU only).

Each pin ties the oracle to something other than itself: the pages' quick
start example (tests/golden/quickstart_propagation.json, values derived by
hand and cited there), the plain operators on sliced inputs, brute force
with numpy, closed forms (one-hot weights, single-point clouds, x = y), exact
integer arithmetic, and float64 references within a rounding bound.
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "quickstart_propagation.json")
U = 2.0 ** -24


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def cloud(seed, B, N, grid=None):
    rng = np.random.default_rng(seed)
    x = rng.random((B, N, 3), dtype=np.float32)
    if grid:
        x = (np.floor(x / grid) * grid).astype(np.float32)
    return x


# --- quick start -----------------------------------------------------------
def test_quickstart_three_nn(oracle_mod):
    g = golden()
    xyz = np.array(g["xyz"], np.float32)
    d, i = oracle_mod.knn_masked(xyz[:, :2], xyz, 3, squared=True)
    assert i.reshape(1, 2, 3).tolist() == g["three_nn"]["idx"]
    assert d.reshape(1, 2, 3).tolist() == g["three_nn"]["dist_squared"]
    d2, i2 = oracle_mod.knn_masked(xyz[:, :2], xyz, 3)
    assert np.array_equal(d2, np.sqrt(d).astype(np.float32))


def test_quickstart_three_interpolate(oracle_mod):
    g = golden()
    idx = np.array(g["three_nn"]["idx"], np.int64)
    f = np.ones((1, 2, 3), np.float32)
    w = np.full((1, 2, 3), np.float32(1.0 / 3.0), np.float32)
    out = oracle_mod.three_interpolate(f, idx, w)
    assert out.tolist() == g["three_interpolate"]["out"]


def test_quickstart_chamfer(oracle_mod):
    g = golden()
    xyz = np.array(g["xyz"], np.float32)
    loss, _, _ = oracle_mod.chamfer(xyz[:, :2], xyz)
    assert loss == np.float32(g["chamfer"]["loss"])


# --- masked kNN / Ball Query ------------------------------------------------
def test_knn_masked_full_lengths_equals_knn(oracle_mod):
    q, x = cloud(1, 2, 20), cloud(2, 2, 50)
    d, i = oracle_mod.knn_masked(q, x, 7, [20, 20], [50, 50])
    wd, wi = oracle_mod.knn(q, x, 7)
    assert np.array_equal(i, wi) and np.array_equal(d, wd)


def test_knn_masked_equals_knn_on_sliced_clouds(oracle_mod):
    q, x = cloud(3, 3, 16, 1 / 8), cloud(4, 3, 40, 1 / 8)
    ql, rl = [16, 5, 0], [40, 3, 12]
    k = 6
    d, i = oracle_mod.knn_masked(q, x, k, ql, rl, squared=True)
    d, i = d.reshape(3, 16, k), i.reshape(3, 16, k)
    for b in range(3):
        nq, nr = ql[b], rl[b]
        assert (i[b, nq:] == -1).all() and (d[b, nq:] == 0).all()
        if nq == 0:
            continue
        kk = min(k, nr)
        if kk > 0:
            wd, wi = oracle_mod.knn(q[b:b + 1, :nq].copy(),
                                    x[b:b + 1, :nr].copy(), kk)
            assert np.array_equal(i[b, :nq, :kk], wi)
            assert np.array_equal(np.sqrt(d[b, :nq, :kk]).astype(np.float32), wd)
        assert (i[b, :nq, kk:] == -1).all() and (d[b, :nq, kk:] == 0).all()


def test_knn_masked_squared_is_s32_of_the_pair(oracle_mod):
    q, x = cloud(5, 1, 30), cloud(6, 1, 64)
    d, i = oracle_mod.knn_masked(q, x, 5, squared=True)
    pairs_q = np.repeat(q[0], 5, axis=0)
    pairs_x = x[0][i.reshape(-1)]
    assert np.array_equal(d.reshape(-1), oracle_mod.s32(pairs_q, pairs_x))


def test_knn_masked_brute_force_lexsort(oracle_mod):
    q, x = cloud(7, 2, 9, 1 / 4), cloud(8, 2, 33, 1 / 4)
    rl = [33, 20]
    d, i = oracle_mod.knn_masked(q, x, 8, None, rl, squared=True)
    for b in range(2):
        for a in range(9):
            xs = x[b, :rl[b]].astype(np.float64)
            s = ((q[b, a].astype(np.float64) - xs) ** 2).sum(1)  # exact on the 1/4 lattice
            order = np.lexsort((np.arange(rl[b]), s))[:8]
            assert i[b * 9 + a].tolist() == order.tolist()


def test_ball_query_masked_equals_sliced(oracle_mod):
    q, x = cloud(9, 3, 12, 1 / 8), cloud(10, 3, 60, 1 / 8)
    ql, rl = [12, 4, 0], [60, 0, 7]
    # r = 0.5: R2 = 0.25 exactly, hit by lattice distances (strictness)
    d, i = oracle_mod.ball_query_masked(q, x, 0.5, 9, ql, rl)
    d, i = d.reshape(3, 12, 9), i.reshape(3, 12, 9)
    for b in range(3):
        nq, nr = ql[b], rl[b]
        assert (i[b, nq:] == -1).all() and (d[b, nq:] == 0).all()
        if nq:
            wd, wi = oracle_mod.ball_query(q[b:b + 1, :nq].copy(),
                                           x[b:b + 1, :nr].copy(), 0.5, 9)
            assert np.array_equal(i[b, :nq], wi) and np.array_equal(d[b, :nq], wd)


def test_gather_points_matches_fancy_indexing(oracle_mod):
    x = cloud(11, 2, 10)
    idx = np.array([[[0, 9, -1], [3, -1, -1]], [[1, 2, 3], [-1, 5, 9]]], np.int64)
    out = oracle_mod.gather_points(x, idx)
    for b in range(2):
        for a in range(2):
            for t in range(3):
                j = idx[b, a, t]
                want = np.zeros(3, np.float32) if j < 0 else x[b, j]
                assert np.array_equal(out[b, a, t], want)
    with pytest.raises(ValueError):
        oracle_mod.gather_points(x, np.full((2, 1, 1), 10, np.int64))


# --- three_interpolate -------------------------------------------------------
def interp_inputs(seed, B=2, C=5, M=11, n=17):
    rng = np.random.default_rng(seed)
    f = rng.standard_normal((B, C, M)).astype(np.float32)
    idx = rng.integers(0, M, (B, n, 3)).astype(np.int64)
    w = rng.random((B, n, 3)).astype(np.float32)
    return f, idx, w


def dense_weights(idx, w, M):
    """W[b, i, m] = sum of the weights of slot entries pointing at m (float64)."""
    B, n, _ = idx.shape
    W = np.zeros((B, n, M))
    for b in range(B):
        for i in range(n):
            for t in range(3):
                if idx[b, i, t] >= 0:
                    W[b, i, idx[b, i, t]] += float(w[b, i, t])
    return W


def test_three_interpolate_one_hot_is_a_gather(oracle_mod):
    f, idx, _ = interp_inputs(12)
    w = np.zeros(idx.shape, np.float32)
    w[..., 1] = 1.0
    out = oracle_mod.three_interpolate(f, idx, w)
    want = np.take_along_axis(f, idx[:, None, :, 1].repeat(f.shape[1], 1), axis=2)
    assert np.array_equal(out, want)


def test_three_interpolate_within_rounding_bound_of_float64(oracle_mod):
    f, idx, w = interp_inputs(13)
    out = oracle_mod.three_interpolate(f, idx, w).astype(np.float64)
    W = dense_weights(idx, w, f.shape[2])
    exact = np.einsum("bcm,bim->bci", f.astype(np.float64), W)
    mag = np.einsum("bcm,bim->bci", np.abs(f.astype(np.float64)), W)
    # three products and two sums, each rounded once: |err| <= 3u sum|w f|
    assert (np.abs(out - exact) <= 3 * U * mag + 1e-45).all()


def test_three_interpolate_exact_on_small_integers(oracle_mod):
    rng = np.random.default_rng(14)
    f = rng.integers(-8, 9, (2, 3, 7)).astype(np.float32)
    idx = rng.integers(0, 7, (2, 9, 3)).astype(np.int64)
    w = rng.integers(-4, 5, (2, 9, 3)).astype(np.float32) / 4
    out = oracle_mod.three_interpolate(f, idx, w)
    exact = np.einsum("bcm,bim->bci", f.astype(np.float64), dense_weights(idx, w, 7))
    assert np.array_equal(out.astype(np.float64), exact)


def test_three_interpolate_padding_reads_zero(oracle_mod):
    f, idx, w = interp_inputs(15)
    idx2 = idx.copy()
    idx2[:, :, 2] = -1
    w0 = w.copy()
    w0[:, :, 2] = 0
    assert np.array_equal(oracle_mod.three_interpolate(f, idx2, w),
                          oracle_mod.three_interpolate(f, idx, w0))
    bad = idx.copy()
    bad[0, 0, 0] = f.shape[2]
    with pytest.raises(ValueError):
        oracle_mod.three_interpolate(f, bad, w)


def test_three_interpolate_backward_exact_on_small_integers(oracle_mod):
    rng = np.random.default_rng(16)
    g = rng.integers(-8, 9, (2, 3, 9)).astype(np.float32)
    idx = rng.integers(0, 7, (2, 9, 3)).astype(np.int64)
    w = rng.integers(-4, 5, (2, 9, 3)).astype(np.float32) / 4
    gf = oracle_mod.three_interpolate_backward(g, idx, w, 7)
    exact = np.einsum("bci,bim->bcm", g.astype(np.float64), dense_weights(idx, w, 7))
    assert np.array_equal(gf.astype(np.float64), exact)


def test_three_interpolate_backward_is_the_adjoint(oracle_mod):
    f, idx, w = interp_inputs(17, M=13, n=40)
    g = np.random.default_rng(18).standard_normal((2, 5, 40)).astype(np.float32)
    gf = oracle_mod.three_interpolate_backward(g, idx, w, 13).astype(np.float64)
    W = dense_weights(idx, w, 13)
    exact = np.einsum("bci,bim->bcm", g.astype(np.float64), W)
    cnt = np.zeros((2, 13))
    for b in range(2):
        np.add.at(cnt[b], idx[b].reshape(-1), 1)
    mag = np.einsum("bci,bim->bcm", np.abs(g.astype(np.float64)), W)
    # s terms summed in float32: |err| <= s u sum|t| (products and sums)
    assert (np.abs(gf - exact) <= (cnt[:, None, :] + 1) * U * mag + 1e-45).all()
    lhs = (oracle_mod.three_interpolate(f, idx, w).astype(np.float64) * g).sum()
    rhs = (f.astype(np.float64) * gf).sum()
    assert abs(lhs - rhs) <= 1e-4 * (np.abs(f).sum() + np.abs(g).sum())


# --- Chamfer -----------------------------------------------------------------
def brute_nn(a, b):
    """Nearest point of b for every point of a: (s, j), float32 s by numpy."""
    d = a[:, None, :] - b[None, :, :]
    s = (d[..., 0] * d[..., 0] + d[..., 1] * d[..., 1]) + d[..., 2] * d[..., 2]
    j = np.argmin(s, axis=1)  # first minimum = smaller index
    return s[np.arange(len(a)), j], j


def test_chamfer_brute_force_and_reductions(oracle_mod):
    x, y = cloud(20, 3, 14), cloud(21, 3, 9)
    loss, (dx, ix), (dy, iy) = oracle_mod.chamfer(x, y)
    per = []
    for b in range(3):
        sx, jx = brute_nn(x[b], y[b])
        sy, jy = brute_nn(y[b], x[b])
        assert np.array_equal(dx[b], sx) and np.array_equal(ix[b], jx)
        assert np.array_equal(dy[b], sy) and np.array_equal(iy[b], jy)
        per.append(sx.astype(np.float64).mean() + sy.astype(np.float64).mean())
    assert abs(float(loss) - np.mean(per)) <= 2 * U * abs(np.mean(per))
    s_sum, _, _ = oracle_mod.chamfer(x, y, point_reduction="sum", batch_reduction="sum")
    want = sum(dx[b].astype(np.float64).sum() + dy[b].astype(np.float64).sum()
               for b in range(3))
    assert abs(float(s_sum) - want) <= 2 * U * want
    none, _, _ = oracle_mod.chamfer(x, y, batch_reduction="none")
    assert none.shape == (3,)
    assert abs(float(loss) - none.astype(np.float64).mean()) <= 4 * U * float(loss)


def test_chamfer_closed_forms(oracle_mod):
    x = cloud(22, 2, 30)
    loss, _, _ = oracle_mod.chamfer(x, x)
    assert loss == 0.0
    a = np.array([[[0.5, 0.25, 0.0]]], np.float32)
    b = np.array([[[1.5, 0.25, 2.0]]], np.float32)
    loss, _, _ = oracle_mod.chamfer(a, b)
    assert loss == np.float32(2 * (1.0 + 4.0))
    one, _, _ = oracle_mod.chamfer(a, b, single_directional=True)
    assert one == np.float32(5.0)
    w, _, _ = oracle_mod.chamfer(a, b, weights=np.array([0.5], np.float32))
    assert w == np.float32(5.0)


def test_chamfer_lengths_equal_sliced_clouds(oracle_mod):
    x, y = cloud(23, 3, 12), cloud(24, 3, 10)
    xl, yl = [12, 5, 0], [10, 2, 4]
    per, (dx, ix), (dy, iy) = oracle_mod.chamfer(x, y, xl, yl, batch_reduction="none")
    for b in range(3):
        if xl[b] == 0:
            assert (ix[b] == -1).all() and (dx[b] == 0).all()
            assert (iy[b] == -1).all()
            assert per[b] == np.float32(0.0)
            continue
        want, _, _ = oracle_mod.chamfer(x[b:b + 1, :xl[b]].copy(),
                                        y[b:b + 1, :yl[b]].copy(),
                                        batch_reduction="none")
        assert per[b] == want[0]
        assert (ix[b, xl[b]:] == -1).all() and (dy[b, yl[b]:] == 0).all()


def test_chamfer_is_symmetric(oracle_mod):
    x, y = cloud(25, 2, 17), cloud(26, 2, 23)
    a, _, _ = oracle_mod.chamfer(x, y)
    b, _, _ = oracle_mod.chamfer(y, x)
    assert a == b
