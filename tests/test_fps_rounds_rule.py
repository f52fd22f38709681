"""CPU pin of the rule by which the FPS rounds kernels certify several
centers per exchange (``fps_rounds_kernel`` and ``fps_grid_rounds_kernel``
in ``csrc/pc_fps.cu``), restated in numpy and compared with the oracle.

The operator (mps-pointops project page, "Farthest point sampling"): each
step takes the point with the largest m_j = min over the centers so far of
s32(x_j, c), the smallest index on an exact tie.  A round certifies a run:

* thread t of block r holds points lo_r + p T + t (p < PPT); a lane's best
  point (largest m, smallest index) and its second largest m; a warp lists
  its best point, then up to FR_CW - 1 lanes whose best is above the warp's
  bound (the largest second m of its lanes, raised to the m of the lanes
  past FR_CW - 1 that are above it);
* CLUSTER: B is the largest bound; the candidates are the first center (the
  largest listed point) and, in list order, the listed points above B, the
  first CAP of them (those past CAP raise B to their m);
* GRID: each cluster's summary is its largest listed point, then its listed
  points above Bc; where more than CAP - 1 lie above the bound, a bound tau
  from two levels of a 64-bin histogram of their keys drops the smallest
  (the same rule picks the cloud's candidates from the summaries);
* the run: the first center is the largest candidate; the candidates' m are
  lowered by each center; the next center is the largest candidate while
  its m is strictly above B, at most RMAX centers.
Every accepted center must be the step-by-step rule's.  The clouds are tie
heavy (lattices, duplicates); the rule is also run with caps of 4 to 16
candidates (it is exact for any cap), so that the histogram bound and the
list-order cap are taken in most rounds; the planted-mistake tests weaken
one step of the rule and show that the comparison with the oracle catches
it.
"""
import numpy as np
import pytest

import oracle
from point_cloud_neighbor_gb300 import inputs

f32 = np.float32
FR_CW, CAP, RMAX = 8, 128, 64
HIST_USED = [0]  # times the histogram bound was taken (the tests check it is)


def s32(x, c):
    d = (x - c).astype(f32)
    sq = (d * d).astype(f32)
    return ((sq[:, 0] + sq[:, 1]).astype(f32) + sq[:, 2]).astype(f32)


def keys(m):
    """bits(m) + 1 for m >= 0 (0 = no point), as int64."""
    return m.view(np.uint32).astype(np.int64) + 1


def warp_lists(m, N, nblocks, T, mutant=None):
    """Per warp: its listed (key, j) entries in list order and its bound."""
    chunk = -(-N // nblocks)
    ppt = -(-chunk // T)
    out = []
    for r in range(nblocks):
        lo, hi = r * chunk, min(N, (r + 1) * chunk)
        for w in range(T // 32):
            lb = np.zeros(32, np.int64)      # lane best key
            lj = np.full(32, 1 << 40, np.int64)
            ls = np.zeros(32, np.int64)      # lane second key
            for lane in range(32):
                t = w * 32 + lane
                js = [lo + p * T + t for p in range(ppt) if lo + p * T + t < hi]
                if not js:
                    continue
                kk = keys(m[js])
                order = sorted(range(len(js)), key=lambda i: (-kk[i], js[i]))
                lb[lane], lj[lane] = kk[order[0]], js[order[0]]
                if len(js) > 1:
                    ls[lane] = kk[order[1]]
            wh = lb.max()
            if wh == 0:
                out.append(([], 0))
                continue
            wl = min((lj[l], l) for l in range(32) if lb[l] == wh)[1]
            bw = ls.max()
            cand = [l for l in range(32) if lb[l] > bw and l != wl]
            over = cand[FR_CW - 1:]
            if over and mutant != "no_overflow_raise":
                bw = max(bw, lb[over].max())
            ents = [(lb[wl], lj[wl])] + [(lb[l], lj[l]) for l in cand[:FR_CW - 1]]
            out.append((ents, bw))
    return out


def cap_bound(kk, bnd, cap=CAP):
    """The two-level histogram bound of fr_cap_bound: the lowest tau it finds
    with at most CAP - 1 of the keys kk (all > bnd) above it."""
    kmax = int(kk.max())
    lo = bnd + 1
    span = kmax - bnd
    s1 = max(0, int(span - 1).bit_length() - 6)
    s2 = max(0, s1 - 6)

    def first_fit(hist, extra):
        cum = np.cumsum(hist[::-1])[::-1] + extra
        ok = np.nonzero(cum <= cap - 1)[0]
        b = int(ok[0]) if len(ok) else 64
        return b, (int(cum[b]) if b < 64 else extra)

    h1 = np.bincount((kk - lo) >> s1, minlength=64)[:64]
    b, cb = first_fit(h1, 0)
    base2 = (b - 1) << s1
    sel = ((kk - lo) >> s1) == b - 1
    h2 = np.bincount(((kk[sel] - lo) - base2) >> s2, minlength=64)[:64]
    c, _ = first_fit(h2, cb)
    return min(lo + base2 + (c << s2) - 1, kmax)


def pick_candidates(entries, bnd, histogram, mutant=None, cap=CAP):
    """entries: (key, j) in list order.  Returns (first, candidates, bound)."""
    first = max(entries, key=lambda e: (e[0], -e[1]))
    above = [e for e in entries if e[0] > bnd]
    if len(above) > cap - 1 and histogram:
        HIST_USED[0] += 1
        tau = cap_bound(np.array([e[0] for e in above], np.int64), bnd, cap)
        if mutant != "no_tau_raise":
            bnd = max(bnd, tau)
        above = [e for e in above if e[0] > tau]
    elif len(above) > cap - 1:
        if mutant != "no_overflow_raise":
            bnd = max(bnd, max(e[0] for e in above[cap - 1:]))
        above = above[:cap - 1]
    return first, above, bnd


def run_of(x, first, cands, bnd, limit, mutant=None):
    pool = {first[1]: first[0]}
    for k, j in cands:
        pool[j] = k
    out = []
    while len(out) < limit and pool:
        kmax = max(pool.values())
        j = min(jj for jj, kk in pool.items() if kk == kmax)
        if out and (kmax < bnd if mutant == "ties_pass" else kmax <= bnd):
            break
        out.append(j)
        js = np.array(list(pool.keys()))
        mm = np.minimum(((np.array(list(pool.values())) - 1).astype(np.uint32)).view(f32),
                        s32(x[js], x[j]))
        pool = dict(zip(js.tolist(), keys(mm.astype(f32)).tolist()))
    return out


def fps_rounds(x, npoint, start, nblocks, T, cs=None, mutant=None, cap=CAP):
    """The CLUSTER rule (cs None: one cluster of nblocks blocks) or the
    two-level GRID rule (clusters of cs blocks); `cap` the candidates a list
    of summaries or a run holds (the kernels' 128; the rule is exact for
    any)."""
    N = x.shape[0]
    m = np.full(N, np.inf, f32)
    out = [start]
    centers = [start]
    while len(out) < npoint:
        for c in centers:
            m = np.minimum(m, s32(x, x[c]))
        lists = warp_lists(m, N, nblocks, T, mutant)
        wpb = T // 32
        if cs is None:
            ents = [e for ls, _ in lists for e in ls]
            bnd = max(b for _, b in lists)
            first, cands, bnd = pick_candidates(ents, bnd, False, mutant, cap)
        else:
            summ, bounds = [], []
            for cl in range(nblocks // cs):
                part = lists[cl * cs * wpb:(cl + 1) * cs * wpb]
                ents = [e for ls, _ in part for e in ls]
                bc = max(b for _, b in part)
                if not ents:
                    bounds.append(bc)
                    continue
                f, ab, bc = pick_candidates(ents, bc, True, mutant, cap)
                summ += [f] + [e for e in ab if e != f]
                bounds.append(bc)
            first, cands, bnd = pick_candidates(summ, max(bounds), True, mutant, cap)
        cands = [e for e in cands if e != first]
        centers = run_of(x, first, cands, bnd, min(RMAX, npoint - len(out)), mutant)
        out += centers
    return np.array(out[:npoint])


def clouds():
    rng = np.random.default_rng(20260)
    lat = (rng.integers(0, 12, (1, 3000, 3)) / 12).astype(f32)
    dup = rng.random((40, 3)).astype(f32)[rng.integers(0, 40, (1, 2048))]
    mix = inputs.large(seed=7, N=4000)
    return [("lattice", lat, 900), ("duplicates", dup, 120), ("mixture", mix, 1200)]


SCHEDULES = [("cluster 4 x 64", 4, 64, None), ("cluster 3 x 96", 3, 96, None),
             ("cluster 8 x 128", 8, 128, None),
             ("grid 2 x 2 x 64", 4, 64, 2), ("grid 4 x 1 x 96", 4, 96, 1),
             ("grid 2 x 4 x 128", 8, 128, 4)]


@pytest.mark.parametrize("cloud", range(3))
@pytest.mark.parametrize("sched", SCHEDULES, ids=[s[0] for s in SCHEDULES])
def test_rounds_rule_equals_the_step_rule(cloud, sched):
    name, x, npoint = clouds()[cloud]
    _, nblocks, T, cs = sched
    want = oracle.fps(x, npoint, 0)[0]
    got = fps_rounds(x[0], npoint, 0, nblocks, T, cs)
    assert np.array_equal(got, want), f"{name}: first difference at {np.argmax(got != want)}"


@pytest.mark.parametrize("cloud", range(3))
@pytest.mark.parametrize("cap", [4, 8, 16])
def test_histogram_bound_with_small_caps(cloud, cap):
    """The same rules with summaries and runs of `cap` candidates, so that
    the histogram bound (and the list-order cap of the one-level rule) is
    taken in most rounds: the samples are still the oracle's."""
    name, x, npoint = clouds()[cloud]
    want = oracle.fps(x, npoint, 0)[0]
    HIST_USED[0] = 0
    got = fps_rounds(x[0], npoint, 0, 4, 64, 2, cap=cap)
    assert np.array_equal(got, want), f"{name}, grid, cap {cap}"
    assert HIST_USED[0] > 0
    got = fps_rounds(x[0], npoint, 0, 4, 64, None, cap=cap)
    assert np.array_equal(got, want), f"{name}, cluster, cap {cap}"


def test_histogram_bound_must_raise_the_bound():
    """Dropping the smallest candidates without raising the bound to tau
    gives a different sample."""
    bad = 0
    for name, x, npoint in clouds():
        got = fps_rounds(x[0], npoint, 0, 4, 64, 2, "no_tau_raise", cap=16)
        bad += int(not np.array_equal(got, oracle.fps(x, npoint, 0)[0]))
    assert bad > 0


@pytest.mark.parametrize("mutant,sched", [
    ("ties_pass", SCHEDULES[0]), ("no_overflow_raise", SCHEDULES[0]),
    ("ties_pass", SCHEDULES[3]),
])
def test_planted_mistakes_are_caught(mutant, sched):
    """A weakened rule (a tie with the bound accepted; an overflow that does
    not raise the bound) gives a different sample on some cloud."""
    _, nblocks, T, cs = sched
    bad = 0
    for name, x, npoint in clouds():
        want = oracle.fps(x, npoint, 0)[0]
        got = fps_rounds(x[0], npoint, 0, nblocks, T, cs, mutant)
        bad += int(not np.array_equal(got, want))
    assert bad > 0, mutant
