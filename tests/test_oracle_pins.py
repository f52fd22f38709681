"""Pins that tie the oracle to the pages and to mathematics, not to itself.

Each test names what it pins:
  * the worked example printed on the mps-pointops project page ("Quick
    start", "Minimal example"), stored under tests/golden/;
  * exact rational arithmetic with binary32 rounding per operation (the
    pages' non-contracted distance order), and the real-valued error bound;
  * closed forms (1-D uniform grid FPS) and independent algorithms (interval
    bisection FPS, Python's sort for kNN, numpy nonzero for Ball Query);
  * invariants and degenerate cases of the three definitions.
A plausible mistake in the oracle (a dropped term, FMA contraction, a wrong
tie rule, <= instead of <, the radius squared in double, a wrong start or
padding value) makes at least one of these fail; see test_oracle_mutants.py.
"""
import heapq
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from _exact import F, round_f32, s32_exact, s32_fma_variant, s_real
from point_cloud_neighbor_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# worked example (project page, "Minimal example")
# --------------------------------------------------------------------------
def test_worked_example_fps(oracle_mod):
    g = _golden("worked_example.json")
    xyz = np.array(g["xyz"], dtype=np.float32)
    idx = oracle_mod.fps(xyz, g["fps"]["npoint"], g["fps"]["start_idx"])
    assert idx.tolist() == g["fps"]["idx"]


def test_worked_example_knn(oracle_mod):
    g = _golden("worked_example.json")
    xyz = np.array(g["xyz"], dtype=np.float32)
    centers = xyz[:, g["fps"]["idx"][0]]
    d, i = oracle_mod.knn(centers, xyz, g["knn"]["k"])
    assert i.reshape(1, 2, 2).tolist() == g["knn"]["idx"]
    assert d.reshape(1, 2, 2).tolist() == g["knn"]["dist"]


def test_worked_example_ball_query(oracle_mod):
    g = _golden("worked_example.json")
    xyz = np.array(g["xyz"], dtype=np.float32)
    centers = xyz[:, g["fps"]["idx"][0]]
    bq = g["ball_query"]
    d2, i = oracle_mod.ball_query(centers, xyz, bq["radius"], bq["K"])
    assert i.reshape(1, 2, 2).tolist() == bq["idx"]
    assert d2.reshape(1, 2, 2).tolist() == bq["dist2"]


# --------------------------------------------------------------------------
# squared distance: exact arithmetic, per-operation rounding, error bound
# --------------------------------------------------------------------------
def _distance_cases(n=400, seed=11):
    rng = np.random.default_rng(seed)
    cases = []
    # ordinary magnitudes
    a = rng.uniform(-1, 1, (n, 3)).astype(np.float32)
    b = rng.uniform(-1, 1, (n, 3)).astype(np.float32)
    cases.append((a, b))
    # close pairs (cancellation in the subtraction)
    c = (a + rng.uniform(-1e-3, 1e-3, (n, 3))).astype(np.float32)
    cases.append((a, c))
    # tiny coordinates: squares land in the subnormal range
    t = (rng.uniform(-1, 1, (n, 3)) * 1e-21).astype(np.float32)
    u = (rng.uniform(-1, 1, (n, 3)) * 1e-21).astype(np.float32)
    cases.append((t, u))
    return cases


def test_s32_matches_exact_per_operation_rounding(oracle_mod):
    for a, b in _distance_cases():
        got = oracle_mod.s32(a, b)
        want = np.array([s32_exact(a[i], b[i]) for i in range(len(a))],
                        dtype=np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_s32_is_not_fma_contracted(oracle_mod):
    """The cases above contain pairs where an FMA-contracted sum differs, so
    the previous test would catch contraction."""
    a, b = _distance_cases()[0]
    differs = sum(s32_exact(a[i], b[i]) != s32_fma_variant(a[i], b[i])
                  for i in range(len(a)))
    assert differs > 0
    got = oracle_mod.s32(a, b)
    fma = np.array([s32_fma_variant(a[i], b[i]) for i in range(len(a))],
                   dtype=np.float32)
    assert not np.array_equal(got, fma)


def test_s32_error_bound_against_real_distance(oracle_mod):
    """|s32 - s| <= ((1+u)^3 - 1) * s + ... for normal results: with u = 2^-24
    and five roundings on non-negative terms the relative error is below 6u
    plus the subtraction error, which is bounded by 2u + u^2 per squared term
    (relative).  8u is a safe bound for results in the normal range."""
    u = Fraction(1, 2 ** 24)
    a, b = _distance_cases()[0]
    got = oracle_mod.s32(a, b)
    for i in range(len(a)):
        s = s_real(a[i], b[i])
        if s == 0:
            assert got[i] == 0
            continue
        err = abs(F(got[i]) - s)
        assert err <= 8 * u * s


def test_s32_symmetric_and_zero(oracle_mod):
    a, b = _distance_cases()[1]
    assert np.array_equal(oracle_mod.s32(a, b), oracle_mod.s32(b, a))
    assert np.all(oracle_mod.s32(a, a) == 0)


# --------------------------------------------------------------------------
# Ball Query threshold and boundary (numerical contracts page)
# --------------------------------------------------------------------------
def test_radius_threshold_is_float32_square_of_float32_radius(oracle_mod):
    found = 0
    rng = np.random.default_rng(5)
    for r in rng.uniform(1e-3, 10.0, 2000):
        want = round_f32(F(np.float32(r)) * F(np.float32(r)))
        got = oracle_mod.radius_threshold(r)
        assert got == want
        if round_f32(Fraction(float(r)) * Fraction(float(r))) != want:
            found += 1
    # the double-precision square (the flat torch_cluster threshold) differs
    # for some radii, so this pin separates the two readings
    assert found > 0


def test_ball_query_boundary_strict(oracle_mod):
    """A reference at exactly s32 == R2 is rejected; one float below is kept."""
    r = 0.5
    R2 = oracle_mod.radius_threshold(r)
    assert R2 == np.float32(0.25)
    below = np.nextafter(np.float32(0.5), np.float32(0))
    q = np.zeros((1, 1, 3), np.float32)
    x = np.array([[[0.5, 0, 0], [below, 0, 0], [0, 0.5, 0], [0, 0, -0.5]]],
                 np.float32)
    d2, i = oracle_mod.ball_query(q, x, r, 4)
    assert i.tolist() == [[1, -1, -1, -1]]
    assert d2[0, 0] == s32_exact(q[0, 0], x[0, 1]) and d2[0, 0] < R2
    assert d2[0, 1:].tolist() == [0, 0, 0]


def test_ball_query_threshold_not_double_square(oracle_mod):
    """Find a radius where fl32(r*r) (double product) and fl32(fl32(r)^2)
    differ, place a point between them, and check the float32 reading."""
    rng = np.random.default_rng(9)
    for r in rng.uniform(0.01, 1.0, 5000):
        r = float(r)
        t32 = round_f32(F(np.float32(r)) * F(np.float32(r)))
        t64 = round_f32(Fraction(r) * Fraction(r))
        if t32 != t64:
            break
    else:
        pytest.fail("no radius separating the two thresholds")
    lo, hi = min(t32, t64), max(t32, t64)
    # a point on the x axis whose s32 equals lo exactly, if one exists; else
    # the largest s32 below hi
    q = np.zeros((1, 1, 3), np.float32)
    a = np.float32(np.sqrt(np.float64(lo)))
    best = None
    for cand in [np.nextafter(a, np.float32(0)), a, np.nextafter(a, np.float32(2))]:
        s = s32_exact([0, 0, 0], [cand, 0, 0])
        if s == lo:
            best = cand
    if best is None:
        pytest.skip("no float32 x with x*x exactly on the lower threshold")
    x = np.array([[[best, 0, 0]]], np.float32)
    _, i = oracle_mod.ball_query(q, x, r, 1)
    accepted = i[0, 0] == 0
    # s32 == lo: accepted iff lo < threshold, i.e. iff the threshold is hi
    assert accepted == (t32 == hi)


def test_ball_query_k_equals_n_is_nonzero(oracle_mod):
    for seed in range(5):
        x = inputs.random_cloud(seed, 2, 40, grid=1 / 16)
        q = inputs.random_cloud(seed + 100, 2, 7, grid=1 / 16)
        r = 0.6
        d2, idx = oracle_mod.ball_query(q, x, r, 40)
        R2 = round_f32(F(np.float32(r)) * F(np.float32(r)))
        for b in range(2):
            for i in range(7):
                s = np.array([s32_exact(q[b, i], x[b, j]) for j in range(40)],
                             np.float32)
                hits = np.nonzero(s < R2)[0]
                row = b * 7 + i
                assert idx[row, :len(hits)].tolist() == hits.tolist()
                assert np.all(idx[row, len(hits):] == -1)
                assert np.array_equal(d2[row, :len(hits)], s[hits])
                assert np.all(d2[row, len(hits):] == 0)


def test_ball_query_first_k_in_input_order(oracle_mod):
    x = inputs.random_cloud(3, 1, 64, grid=1 / 8)
    q = x[:, :5]
    for K in (1, 3, 7):
        _, idx = oracle_mod.ball_query(q, x, 0.7, K)
        _, full = oracle_mod.ball_query(q, x, 0.7, 64)
        for r in range(5):
            hits = [j for j in full[r] if j >= 0]
            want = hits[:K] + [-1] * (K - min(K, len(hits)))
            assert idx[r].tolist() == want


def test_ball_query_empty_reference(oracle_mod):
    q = inputs.random_cloud(0, 2, 3)
    x = np.zeros((2, 0, 3), np.float32)
    d2, idx = oracle_mod.ball_query(q, x, 0.5, 4)
    assert np.all(idx == -1) and np.all(d2 == 0)


def test_ball_query_nan_reference_never_accepted(oracle_mod):
    q = np.zeros((1, 1, 3), np.float32)
    x = np.array([[[np.nan, 0, 0], [0.1, 0, 0]]], np.float32)
    _, idx = oracle_mod.ball_query(q, x, 1.0, 2)
    assert idx.tolist() == [[1, -1]]


# --------------------------------------------------------------------------
# kNN: exact (s, j) order by Python's sort; k = N is the full lexsort
# --------------------------------------------------------------------------
def _knn_exact(q, x, k):
    keys = sorted((s32_exact(q, x[j]), j) for j in range(len(x)))[:k]
    idx = [j for _, j in keys]
    # sqrt of a float32 computed in double then rounded to float32 is the
    # correctly rounded float32 sqrt (53 >= 2*24 + 2)
    dist = [np.float32(np.sqrt(np.float64(s))) for s, _ in keys]
    return dist, idx


@pytest.mark.parametrize("seed,grid", [(0, None), (1, 1 / 8), (2, 1 / 4)])
def test_knn_matches_exact_sort(oracle_mod, seed, grid):
    B, Q, N, k = 2, 6, 33, 9
    x = inputs.random_cloud(seed, B, N, grid=grid)
    q = inputs.random_cloud(seed + 50, B, Q, grid=grid)
    d, i = oracle_mod.knn(q, x, k)
    for b in range(B):
        for t in range(Q):
            dist, idx = _knn_exact(q[b, t], x[b], k)
            assert i[b * Q + t].tolist() == idx
            assert np.array_equal(d[b * Q + t], np.array(dist, np.float32))


def test_knn_k_equals_n_is_full_lexsort(oracle_mod):
    x = inputs.random_cloud(4, 1, 50, grid=1 / 4)
    q = inputs.random_cloud(5, 1, 4, grid=1 / 4)
    d, i = oracle_mod.knn(q, x, 50)
    for t in range(4):
        s = np.array([s32_exact(q[0, t], x[0, j]) for j in range(50)],
                     np.float32)
        order = np.lexsort((np.arange(50), s))
        assert i[t].tolist() == order.tolist()
    assert np.all(np.sort(i, axis=1) == np.arange(50))


def test_knn_duplicate_ties_go_to_smaller_index(oracle_mod):
    x = np.array([[[1, 0, 0], [0, 0, 0], [1, 0, 0], [0, 0, 0], [0, 2, 0]]],
                 np.float32)
    q = np.zeros((1, 1, 3), np.float32)
    d, i = oracle_mod.knn(q, x, 4)
    assert i.tolist() == [[1, 3, 0, 2]]
    assert d.tolist() == [[0, 0, 1, 1]]


def test_knn_rows_sampling_consistent(oracle_mod):
    x = inputs.random_cloud(7, 3, 40)
    q = inputs.random_cloud(8, 3, 10)
    d, i = oracle_mod.knn(q, x, 5)
    rows = np.array([0, 13, 29], np.int64)
    ds, is_ = oracle_mod.knn(q, x, 5, rows=rows)
    assert np.array_equal(is_, i[rows]) and np.array_equal(ds, d[rows])
    dt, it = oracle_mod.knn(q, x, 5, threads=3)
    assert np.array_equal(it, i) and np.array_equal(dt, d)


def test_knn_rejects_k_above_n(oracle_mod):
    x = inputs.random_cloud(0, 1, 4)
    with pytest.raises(ValueError):
        oracle_mod.knn(x, x, 5)


# --------------------------------------------------------------------------
# FPS: closed form on a 1-D grid, interval bisection, brute force, invariants
# --------------------------------------------------------------------------
def _line(n):
    x = np.zeros((1, n, 3), np.float32)
    x[0, :, 0] = np.arange(n, dtype=np.float32)
    return x


@pytest.mark.parametrize("L", [2, 3, 4, 5])
def test_fps_uniform_grid_closed_form(oracle_mod, L):
    """n = 2^L + 1 points 0..n-1 on a line, start 0: the far end, then at each
    level the odd multiples of (n-1)/2^l in increasing order."""
    n = 2 ** L + 1
    want = [0, n - 1]
    for lev in range(1, L + 1):
        step = (n - 1) >> lev
        want += [m * step for m in range(1, 2 ** lev, 2)]
    got = oracle_mod.fps(_line(n), n, 0)
    assert got[0].tolist() == want


def _fps_by_intervals(n, start, npoint):
    """FPS on integer points 0..n-1 of a line by interval bisection: keep the
    gaps between selected points in a heap keyed by (-distance of the gap's
    farthest point, that point's index).  Independent of scanning all points."""
    out = [start]
    heap = []
    if start > 0:
        heap.append((-(start ** 2), 0, "left", 0, start))
    if start < n - 1:
        heap.append((-((n - 1 - start) ** 2), n - 1, "right", start, n - 1))
    heapq.heapify(heap)
    while len(out) < npoint:
        if not heap:
            out.append(0)           # every point taken: the rule yields j = 0
            continue
        _, j, kind, a, b = heapq.heappop(heap)
        out.append(j)
        # split the segment at j into the parts still containing points
        segs = []
        if kind == "left":
            segs = [("left", 0, j)] if j > 0 else []
            segs.append(("gap", j, b))
        elif kind == "right":
            segs = [("gap", a, j)]
            if j < n - 1:
                segs.append(("right", j, n - 1))
        else:
            segs = [("gap", a, j), ("gap", j, b)]
        for kind2, a2, b2 in segs:
            if kind2 == "left":
                if b2 > 0:
                    heapq.heappush(heap, (-(b2 ** 2), 0, "left", 0, b2))
            elif kind2 == "right":
                if a2 < n - 1:
                    heapq.heappush(heap, (-((n - 1 - a2) ** 2), n - 1, "right",
                                          a2, n - 1))
            elif b2 - a2 >= 2:
                h = (b2 - a2) // 2
                heapq.heappush(heap, (-(h * h), a2 + h, "gap", a2, b2))
    return out


@pytest.mark.parametrize("n,start", [(23, 0), (23, 7), (40, 39), (13, 6), (9, 0)])
def test_fps_line_matches_interval_bisection(oracle_mod, n, start):
    got = oracle_mod.fps(_line(n), n + 3, start)
    assert got[0].tolist() == _fps_by_intervals(n, start, n + 3)


def _fps_from_scratch(x, npoint, start):
    """Recompute m_j = min over all selected centers from scratch each step."""
    N = len(x)
    s = np.array([[s32_exact(x[a], x[b]) for b in range(N)] for a in range(N)],
                 np.float32)
    sel = [start]
    for _ in range(1, npoint):
        m = s[:, sel].min(axis=1)
        mx = m.max()
        sel.append(int(np.nonzero(m == mx)[0][0]))
    return sel


@pytest.mark.parametrize("seed,grid", [(0, None), (1, 1 / 4), (2, 1 / 2)])
def test_fps_matches_brute_force(oracle_mod, seed, grid):
    x = inputs.random_cloud(seed, 2, 24, grid=grid)
    got = oracle_mod.fps(x, 30, 3)
    for b in range(2):
        assert got[b].tolist() == _fps_from_scratch(x[b], 30, 3)


def test_fps_exhaustion_repeats_zero(oracle_mod):
    x = inputs.random_cloud(3, 1, 5)
    got = oracle_mod.fps(x, 9, 2)[0].tolist()
    assert got[0] == 2 and sorted(got[:5]) == [0, 1, 2, 3, 4]
    assert got[5:] == [0, 0, 0, 0]


def test_fps_duplicates_selected_once_while_distance_positive(oracle_mod):
    x = inputs.tiny()
    idx = oracle_mod.fps(x, 64, 0)[0]
    assert len(set(idx.tolist())) == 64
    assert idx[0] == 0


def test_fps_min_distance_non_increasing(oracle_mod):
    x = inputs.random_cloud(12, 1, 300)[0]
    idx = oracle_mod.fps(x[None], 80, 0)[0]
    prev = np.inf
    for t in range(1, 80):
        m = oracle_mod.min_dist_to_set(x, idx[:t], idx[t:t + 1])[0]
        assert m <= prev
        # and c_t attains the maximum of m over all points (smallest j on ties)
        mall = oracle_mod.min_dist_to_set(x, idx[:t], np.arange(300))
        assert m == mall.max() and idx[t] == np.nonzero(mall == m)[0][0]
        prev = m


def test_fps_rejects_bad_start(oracle_mod):
    x = inputs.random_cloud(0, 1, 4)
    with pytest.raises(ValueError):
        oracle_mod.fps(x, 2, 4)


def test_ball_query_scan_length(oracle_mod):
    """Pairs the first-K rule examines: the K-th accepted index + 1, else N
    (exact s32 and numpy nonzero, independent of the oracle's scan)."""
    x = inputs.random_cloud(31, 2, 60, grid=1 / 8)
    q = inputs.random_cloud(32, 2, 9, grid=1 / 8)
    r, K = 0.7, 5
    R2 = round_f32(F(np.float32(r)) * F(np.float32(r)))
    got = oracle_mod.ball_query_scan_len(q, x, r, K)
    for b in range(2):
        for i in range(9):
            s = np.array([s32_exact(q[b, i], x[b, j]) for j in range(60)], np.float32)
            hits = np.nonzero(s < R2)[0]
            want = hits[K - 1] + 1 if len(hits) >= K else 60
            assert got[b * 9 + i] == want


# --------------------------------------------------------------------------
# the all-core FPS (points of each step split over host threads) is the
# plain FPS: same pins, and equal to it on ties, exhaustion and thread
# counts above the number of points
# --------------------------------------------------------------------------
@pytest.mark.parametrize("threads", [1, 2, 3, 8, 33])
def test_fps_all_cores_equals_plain(oracle_mod, threads):
    cases = [(inputs.random_cloud(40, 3, 500), 120, 7),
             (inputs.random_cloud(41, 2, 300, grid=1 / 4), 310, 0),   # ties, exhausted
             (inputs.tiny(), 64, 0),                                  # duplicates
             (inputs.random_cloud(42, 1, 5), 9, 2)]                   # N < threads
    for x, npoint, start in cases:
        want = oracle_mod.fps(x, npoint, start)
        got = oracle_mod.fps_all_cores(x, npoint, start, threads=threads)
        assert np.array_equal(got, want), (x.shape, npoint, start, threads)


@pytest.mark.parametrize("L", [3, 5])
def test_fps_all_cores_uniform_grid_closed_form(oracle_mod, L):
    n = 2 ** L + 1
    want = [0, n - 1]
    for lev in range(1, L + 1):
        step = (n - 1) >> lev
        want += [m * step for m in range(1, 2 ** lev, 2)]
    got = oracle_mod.fps_all_cores(_line(n), n, 0, threads=4)
    assert got[0].tolist() == want


def test_fps_all_cores_matches_brute_force(oracle_mod):
    x = inputs.random_cloud(1, 2, 24, grid=1 / 4)
    got = oracle_mod.fps_all_cores(x, 30, 3, threads=5)
    for b in range(2):
        assert got[b].tolist() == _fps_from_scratch(x[b], 30, 3)
