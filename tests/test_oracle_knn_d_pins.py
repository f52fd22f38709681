"""Pins of the oracle's D-dimensional kNN (CPU only).

The distance is pinned to exact rational arithmetic with one binary32
rounding per operation in increasing dimension (tests/_exact.py), which
catches a reordered, dropped or contracted term; D = 3 must equal the 3-D
operator; the selection is pinned to a lexsort of exact squared distances on
a dyadic lattice where every distance is exact in float32.
"""
import numpy as np

from _exact import sd_exact


def test_distance_matches_exact_rounding_per_operation(oracle_mod):
    rng = np.random.default_rng(90)
    for D in (1, 2, 5, 17, 64):
        for _ in range(40):
            # mixed magnitudes so that the summation order matters
            a = (rng.standard_normal(D) * 10.0 ** rng.integers(-3, 4, D)).astype(np.float32)
            b = (a + rng.standard_normal(D).astype(np.float32) * np.float32(1e-3)).astype(np.float32)
            assert oracle_mod.sd(a, b) == sd_exact(a, b), D


def test_order_of_accumulation_is_increasing_dimension(oracle_mod):
    # a large term first and many small ones after: the small ones vanish only
    # when added one by one after the large one (reversed order keeps them)
    a = np.array([2048.0] + [0.0] * 8, np.float32)
    # 2048^2 = 2^22 (ulp 0.5); each 0.25^2 = 0.0625 rounds away when added to
    # it, while the eight of them summed first make 0.5, one ulp
    b = np.array([0.0] + [0.25] * 8, np.float32)
    got = oracle_mod.sd(a, b)
    assert got == sd_exact(a, b)
    rev = sd_exact(a[::-1].copy(), b[::-1].copy())
    assert got != rev


def test_three_dimensions_equal_the_point_operator(oracle_mod):
    rng = np.random.default_rng(91)
    q = rng.random((2, 30, 3), dtype=np.float32)
    x = rng.random((2, 200, 3), dtype=np.float32)
    d, i = oracle_mod.knn_d(q, x, 9)
    wd, wi = oracle_mod.knn(q, x, 9)
    assert np.array_equal(i, wi) and np.array_equal(d, wd)


def test_selection_on_a_lattice_is_the_exact_lexsort(oracle_mod):
    rng = np.random.default_rng(92)
    D, N, Q, k = 7, 90, 12, 15
    x = (rng.integers(0, 8, (1, N, D)) / 8).astype(np.float32)
    q = (rng.integers(0, 8, (1, Q, D)) / 8).astype(np.float32)
    d, i = oracle_mod.knn_d(q, x, k, squared=True)
    for a in range(Q):
        s = ((q[0, a].astype(np.float64) - x[0].astype(np.float64)) ** 2).sum(1)
        order = np.lexsort((np.arange(N), s))[:k]
        assert i[a].tolist() == order.tolist()
        assert d[a].tolist() == s[order].tolist()
    d2, _ = oracle_mod.knn_d(q, x, k)
    assert np.array_equal(d2, np.sqrt(d).astype(np.float32))
