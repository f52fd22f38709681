"""CPU pin of the candidate filter that every kNN and Ball Query kernel runs
before its exact squared distance (the header of ``csrc/pc_filter.cuh``).

The kernels never decide a selection with the filter: they recompute the
exact s32 of every pair that passes.  So the filter is sound iff no pair
whose s32 meets the selection bound is rejected:

    s32(q, x) <= tau   ==>   t' <= thr                                  (P0)

with, for a frame centre c (any float point),
    x' = fl(x - c), q' = fl(q - c),
    W  = fma(z', z', fma(y', y', fl(x' x')))      (likewise qq for q'),
    w' = fl(W (1 - 2^-17))   (W > 1e30: x' = 0 and w' = -inf),
    a  = -2 q'               (qq > 1e30: a = 0),
    t' = fma(a_z, z', fma(a_y, y', fma(a_x, x', w'))),
    thr = fl(fl(fl(tau (1 + 2^-20)) - fl(qq (1 - 2^-19))) + 2^-120)
          (+inf when qq > 1e30 or tau > 3e38).
This file restates that arithmetic in numpy float32 (every operation one
IEEE rounding; the FMA emulated with one rounding by ``_exact.fma_f32``,
itself pinned here against exact rational arithmetic) and checks, on
adversarial pairs, (P0) and the two steps the header's proof goes through:

    t'  <= B := tau (1 + 6.1u) + 6 * 2^-150 - qq (1 - 11.02u)          (P1)
    thr >= B                                                            (P2)

(u = 2^-24).  Because every operation in thr is monotone in tau, the
tightest case of (P0) is tau = s32 itself, which is what every population
below uses (an exact tie at the bound: kNN keeps s32 == tau, and Ball
Query's strict s32 < R2 means tau = prevfloat(R2) at worst).

The planted-mistake test at the end changes one piece of the restated
arithmetic at a time and shows that (P0)-(P2) catch it.
"""
from fractions import Fraction

import numpy as np
import pytest

from _exact import F, fma_exact, fma_f32, round_f32

f32 = np.float32
INF = f32(np.inf)
U = 2.0 ** -24


# --------------------------------------------------------------------------
# the filter, restated (one float32 rounding per operation)
# --------------------------------------------------------------------------
def _norm2(x, y, z):
    return fma_f32(z, z, fma_f32(y, y, (x * x).astype(f32)))


def filter_eval(q, x, c, tau, mutant=None):
    """Return (t', thr, qq, W) for pair rows q[i], x[i] in the frame c[i]."""
    q = np.asarray(q, f32)
    x = np.asarray(x, f32)
    c = np.broadcast_to(np.asarray(c, f32), q.shape)
    tau = np.asarray(tau, f32)
    with np.errstate(over="ignore", invalid="ignore"):
        xp = (x - c).astype(f32)
        qp = (q - c).astype(f32) if mutant != "query_uncentred" else q.copy()
        W = _norm2(xp[:, 0], xp[:, 1], xp[:, 2])
        shrink = {"drop_shrink": f32(1.0), "shrink_sign": f32(1 + 2 ** -17),
                  "no_slack": f32(1.0)}.get(mutant, f32(1 - 2 ** -17))
        wbig = ~(W <= f32(1e30))
        w = np.where(wbig, -INF, (W * shrink).astype(f32))
        xp = np.where(wbig[:, None], f32(0), xp)
        qq = _norm2(qp[:, 0], qp[:, 1], qp[:, 2])
        qbig = ~(qq <= f32(1e30))
        two = f32(2.0) if mutant == "a_sign" else f32(-2.0)
        a = np.where(qbig[:, None], f32(0), (two * qp).astype(f32))
        t = fma_f32(a[:, 0], xp[:, 0], w)
        t = fma_f32(a[:, 1], xp[:, 1], t)
        t = fma_f32(a[:, 2], xp[:, 2], t)
        up = f32(1.0) if mutant in ("no_slack", "no_tau_qq_slack") else f32(1 + 2 ** -20)
        dn = f32(1.0) if mutant in ("no_slack", "no_tau_qq_slack") else f32(1 - 2 ** -19)
        d = ((tau * up).astype(f32) - (qq * dn).astype(f32)).astype(f32)
        absterm = f32(0.0) if mutant == "no_abs_term" else f32(2 ** -120)
        thr = (d + absterm).astype(f32)
        thr = np.where(qbig | ~(tau <= f32(3e38)), INF, thr).astype(f32)
    return t, thr, qq, W


def s32(q, x):
    """((dx*dx + dy*dy) + dz*dz), one float32 rounding per operation."""
    d = (np.asarray(q, f32) - np.asarray(x, f32)).astype(f32)
    s = (d * d).astype(f32)
    return ((s[:, 0] + s[:, 1]).astype(f32) + s[:, 2]).astype(f32)


def _bound_B(tau, qq):
    """B = tau (1 + 6.1u) + 6 * 2^-150 - qq (1 - 11.02u), as float64 with an
    error far below the u-scale margins (checked exactly where it is close)."""
    return (tau.astype(np.float64) * (1 + 6.1 * U) + 6 * 2.0 ** -150
            - qq.astype(np.float64) * (1 - 11.02 * U))


def _bound_B_exact(tau, qq):
    return (F(tau) * (1 + Fraction(61, 10) * Fraction(1, 2 ** 24)) + 6 * Fraction(1, 2 ** 150)
            - F(qq) * (1 - Fraction(1102, 100) * Fraction(1, 2 ** 24)))


def check_pairs(q, x, c, mutant=None):
    """Counts of rows violating (P0), (P1), (P2) with tau = s32(q, x)."""
    tau = s32(q, x)
    t, thr, qq, W = filter_eval(q, x, c, tau, mutant)
    fin = np.isfinite(tau)
    assert not np.isnan(t[fin]).any(), "t' must never be NaN for finite coordinates"
    p0 = fin & ~(t <= thr)
    guarded = ~(W <= f32(1e30)) | ~(qq <= f32(1e30))
    B = _bound_B(tau, qq)
    scale = U * (np.abs(W.astype(np.float64)) + np.abs(qq.astype(np.float64))
                 + np.abs(tau.astype(np.float64))) + 2.0 ** -140
    p1 = fin & ~guarded & (t.astype(np.float64) > B + 1e-9 * scale)
    p2 = fin & ~guarded & (thr.astype(np.float64) < B - 1e-9 * scale)
    # rows within float64 noise of B are decided exactly
    near1 = fin & ~guarded & ~p1 & (np.abs(t.astype(np.float64) - B) <= 1e-9 * scale)
    near2 = fin & ~guarded & ~p2 & (np.abs(thr.astype(np.float64) - B) <= 1e-9 * scale)
    for i in np.nonzero(near1)[0]:
        if F(t[i]) > _bound_B_exact(tau[i], qq[i]):
            p1[i] = True
    for i in np.nonzero(near2)[0]:
        if F(thr[i]) < _bound_B_exact(tau[i], qq[i]):
            p2[i] = True
    return int(p0.sum()), int(p1.sum()), int(p2.sum())


# --------------------------------------------------------------------------
# adversarial populations (seeded)
# --------------------------------------------------------------------------
def _frames_of(cloud):
    """The kernels' frame centres: bounding-box centre of the first 256
    points, and of 256 points spread evenly over the cloud."""
    out = []
    for pts in (cloud[:256], cloud[:: max(1, len(cloud) // 256)][:256]):
        lo, hi = pts.min(axis=0), pts.max(axis=0)
        out.append(((lo + hi).astype(f32) * f32(0.5)).astype(f32))
    return out


def _mixture(rng, n):
    means = rng.random((64, 3))
    pick = rng.integers(0, 64, n)
    return (means[pick] + rng.standard_normal((n, 3)) * 0.05).astype(f32)


def populations():
    rng = np.random.default_rng(20240)
    pops = []
    base = _mixture(rng, 20000)
    morton_like = base[np.lexsort((base[:, 2], base[:, 1], base[:, 0]))]
    for off in (0.0, 1e3, 1e5, 3e6):
        for name, cloud in (("random", base), ("sorted", morton_like)):
            pts = (cloud.astype(np.float64) + off).astype(f32)
            n = len(pts)
            i = rng.integers(0, n, 40000)
            # near pairs (neighbour scale) and far pairs within the cloud
            near = (pts[i] + rng.standard_normal((40000, 3)) * 10 ** rng.uniform(-5, -1, (40000, 1))).astype(f32)
            far = pts[rng.integers(0, n, 40000)]
            for c in _frames_of(pts):
                pops.append((f"{name}+{off:g} near", pts[i], near, c))
                pops.append((f"{name}+{off:g} far", pts[i], far, c))
    # geometric search: q' and x' at a length ratio and a small angle, far
    # from the centre (the case where rounding is largest relative to tau)
    for trial in range(24):
        n = 100000
        ratio = 10 ** rng.uniform(-2, 2)
        L = 10 ** rng.uniform(-3, 6)
        ang = 10 ** rng.uniform(-7, 0)
        dq = rng.standard_normal((n, 3))
        dq /= np.linalg.norm(dq, axis=1, keepdims=True)
        dx = dq + rng.standard_normal((n, 3)) * ang
        dx /= np.linalg.norm(dx, axis=1, keepdims=True)
        pops.append((f"geometry {trial}", (dq * L).astype(f32),
                     (dx * L * ratio).astype(f32), np.zeros(3, f32)))
    # neighbours one ulp apart and exact duplicates, far from the centre
    for L in (1e2, 1e5, 1e7):
        q = (rng.standard_normal((40000, 3)) * L).astype(f32)
        x = np.nextafter(q, np.where(rng.random((40000, 3)) < 0.5, np.inf, -np.inf).astype(f32))
        pops.append((f"ulp neighbours {L:g}", q, x, np.zeros(3, f32)))
        pops.append((f"duplicates {L:g}", q, q.copy(), (rng.standard_normal(3) * L).astype(f32)))
    # subnormal squares (coordinates ~1e-21: every square underflows)
    for s in (1e-19, 1e-21, 1e-23, 1e-25):
        q = (rng.random((40000, 3)) * s).astype(f32)
        x = (rng.random((40000, 3)) * s).astype(f32)
        pops.append((f"subnormal {s:g}", q, x, (rng.random(3) * s).astype(f32)))
        pops.append((f"subnormal {s:g} far centre", q, x, (rng.random(3) * s * 1e4).astype(f32)))
        pops.append((f"subnormal {s:g} duplicates", q, q.copy(), np.zeros(3, f32)))
    # around the 1e30 guards: |x'|^2 and |q'|^2 just below and above 1e30
    for g in (0.9, 0.999999, 1.000001, 1.2):
        n = 40000
        d = rng.standard_normal((n, 3))
        d /= np.linalg.norm(d, axis=1, keepdims=True)
        r = np.sqrt(1e30 * g)
        q = (d * r).astype(f32)
        x = (d * r * (1 + rng.standard_normal((n, 1)) * 1e-3)).astype(f32)
        pops.append((f"guard {g}", q, x, np.zeros(3, f32)))
        pops.append((f"guard {g} query near centre", (d * 1e3).astype(f32), x, np.zeros(3, f32)))
    return pops


_POPS = None


def _pops():
    global _POPS
    if _POPS is None:
        _POPS = populations()
    return _POPS


# --------------------------------------------------------------------------
# the emulated FMA is the correctly rounded a*b + c
# --------------------------------------------------------------------------
def test_fma_emulation_is_exact():
    rng = np.random.default_rng(7)
    n = 3000
    a = (rng.standard_normal(n) * np.exp2(rng.integers(-70, 60, n))).astype(f32)
    b = (rng.standard_normal(n) * np.exp2(rng.integers(-70, 60, n))).astype(f32)
    c = (-(a.astype(np.float64) * b) * (1 + rng.standard_normal(n)
                                       * np.exp2(rng.integers(-40, 0, n)))).astype(f32)
    # double-rounding traps: a*b = half an ulp of c times (1 - 2^-46), so the
    # float64 sum lands on a float32 midpoint while the exact sum does not
    m = 400
    r = rng.uniform(1, 2, m).astype(f32)
    ulp = np.spacing(r).astype(np.float64)
    a2 = (rng.choice([-1.0, 1.0], m) * ulp / 2 * (1 + 2 ** -23)).astype(f32)
    b2 = (1 + rng.choice([-1.0, 1.0], m) * 2 ** -23).astype(f32)
    # subnormal results
    a3 = (rng.standard_normal(300) * 2.0 ** -75).astype(f32)
    b3 = (rng.standard_normal(300) * 2.0 ** -75).astype(f32)
    c3 = (rng.standard_normal(300) * 2.0 ** -148).astype(f32)
    A = np.concatenate([a, a2, a3])
    Bv = np.concatenate([b, b2, b3])
    C = np.concatenate([c, r, c3])
    got = fma_f32(A, Bv, C)
    want = np.array([fma_exact(*t) for t in zip(A, Bv, C)], f32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # the traps are real: one rounding of the float64 sum gets some wrong
    naive = (a2.astype(np.float64) * b2 + r).astype(f32)
    assert (naive != want[n:n + m]).sum() > 0


def test_restated_ops_round_once():
    """Spot-check the numpy float32 steps against exact rational rounding."""
    rng = np.random.default_rng(8)
    q = (rng.standard_normal((200, 3)) * 1e3).astype(f32)
    x = (q + rng.standard_normal((200, 3))).astype(f32)
    s = s32(q, x)
    for i in range(200):
        d = [round_f32(F(q[i, a]) - F(x[i, a])) for a in range(3)]
        sq = [round_f32(F(v) * F(v)) for v in d]
        want = round_f32(F(round_f32(F(sq[0]) + F(sq[1]))) + F(sq[2]))
        assert s[i] == want
    n2 = _norm2(q[:, 0], q[:, 1], q[:, 2])
    for i in range(200):
        xx = round_f32(F(q[i, 0]) * F(q[i, 0]))
        want = fma_exact(q[i, 2], q[i, 2], fma_exact(q[i, 1], q[i, 1], xx))
        assert n2[i] == want


# --------------------------------------------------------------------------
# (P0)-(P2) on every population
# --------------------------------------------------------------------------
def test_filter_is_sound_on_adversarial_pairs():
    bad = []
    total = 0
    for name, q, x, c in _pops():
        p0, p1, p2 = check_pairs(q, x, c)
        total += len(q)
        if p0 or p1 or p2:
            bad.append((name, p0, p1, p2))
    assert total > 2_000_000
    assert not bad, f"filter bound violated: {bad[:5]}"


def test_proof_steps_centring_and_distance():
    """The two exact-arithmetic steps of the header's proof on pairs far from
    the centre: s32 >= D^2 (1 - 5u) - 5 * 2^-150, and
    D'^2 <= D^2 (1 + u) + 2.001 u (W + QQ), with D, D', W, QQ exact."""
    rng = np.random.default_rng(9)
    u = Fraction(1, 2 ** 24)
    tiny = Fraction(1, 2 ** 150)
    for L, D in ((1.0, 1e-3), (1e4, 1e-2), (3e6, 1.0), (1e-21, 1e-21)):
        c = (rng.standard_normal(3) * L).astype(f32)
        q = (c + rng.standard_normal((150, 3)) * L).astype(f32)
        x = (q + rng.standard_normal((150, 3)) * D).astype(f32)
        s = s32(q, x)
        xp = (x - c).astype(f32)
        qp = (q - c).astype(f32)
        for i in range(150):
            D2 = sum((F(q[i, a]) - F(x[i, a])) ** 2 for a in range(3))
            assert F(s[i]) >= D2 * (1 - 5 * u) - 5 * tiny
            Dp2 = sum((F(qp[i, a]) - F(xp[i, a])) ** 2 for a in range(3))
            Wv = sum(F(v) ** 2 for v in xp[i])
            QQ = sum(F(v) ** 2 for v in qp[i])
            assert Dp2 <= D2 * (1 + u) + Fraction(2001, 1000) * u * (Wv + QQ)


def test_guards_and_nan():
    """Beyond the 1e30 guards the pair always passes; a NaN coordinate's
    exact s32 is NaN, which no selection rule accepts, and its t' passes
    or not without affecting anything else."""
    q = np.array([[1e16, 0, 0], [0, 0, 0], [3e15, 3e15, 3e15]], f32)
    x = np.array([[0, 0, 0], [2e15, 0, 0], [3e15, 3e15, 3e15]], f32)
    tau = np.array([0.0, 0.0, 0.0], f32)
    t, thr, qq, W = filter_eval(q, x, np.zeros(3, f32), tau)
    assert thr[0] == np.inf                 # query beyond the guard
    assert t[1] == -np.inf                  # reference beyond the guard
    assert (t <= thr).all()
    qn = np.array([[np.nan, 0, 0]], f32)
    assert np.isnan(s32(qn, np.zeros((1, 3), f32))).all()


# --------------------------------------------------------------------------
# planted mistakes: each is caught by (P0), (P1) or (P2) on some population
# --------------------------------------------------------------------------
MUTANTS = {
    "drop_shrink": "w' = fl(W), the (1 - 2^-17) factor dropped",
    "shrink_sign": "w' = fl(W (1 + 2^-17))",
    "no_tau_qq_slack": "thr = fl(tau - qq) + 2^-120 (no 2^-20 / 2^-19 factors)",
    "no_slack": "no relative slack anywhere",
    "no_abs_term": "the 2^-120 term dropped (subnormal pairs)",
    "a_sign": "a = +2 q'",
    "query_uncentred": "q' = q, the query not moved into the frame",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant):
    caught = []
    for name, q, x, c in _pops():
        p0, p1, p2 = check_pairs(q, x, c, mutant)
        if p0 or p1 or p2:
            caught.append((name, p0, p1, p2))
            break
    assert caught, f"planted mistake not caught: {MUTANTS[mutant]}"
