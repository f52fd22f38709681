"""Reference points placed exactly on the Ball Query boundary, found with the
oracle's own arithmetic.

For a radius r the threshold is R2 = fl32(fl32(r)^2) and a reference is
accepted iff its squared distance s32 < R2.  Starting from c + r * u for a
random unit direction u, one coordinate is walked float by float
(nextafter) and every position whose oracle s32 equals R2 exactly (must be
rejected) or equals the float just below R2 (must be accepted) is kept.
"""
import numpy as np

import oracle


def _step(v: np.ndarray, k: int) -> np.ndarray:
    """Move every float32 of v by k representable steps."""
    out = v.copy()
    target = np.float32(np.inf) if k > 0 else np.float32(-np.inf)
    for _ in range(abs(k)):
        out = np.nextafter(out, target)
    return out


def boundary_points(centers: np.ndarray, radius: float, n_each: int, seed: int):
    """Return (reject, accept): lists of (center index, float32 point [3])."""
    R2 = oracle.radius_threshold(radius)
    below = np.nextafter(R2, np.float32(0))
    r32 = float(np.float32(radius))
    rng = np.random.default_rng(seed)
    reject, accept = [], []
    used = set()
    for _ in range(64):
        if len(reject) >= n_each and len(accept) >= n_each:
            break
        m = 4096
        ci = rng.integers(0, len(centers), m)
        u = rng.standard_normal((m, 3))
        u /= np.linalg.norm(u, axis=1, keepdims=True)
        p0 = (centers[ci].astype(np.float64) + r32 * u).astype(np.float32)
        axis = rng.integers(0, 3)
        for k in range(-8, 9):
            p = p0.copy()
            p[:, axis] = _step(p0[:, axis], k)
            s = oracle.s32(centers[ci], p)
            for sel, bucket in ((s == R2, reject), (s == below, accept)):
                for t in np.nonzero(sel)[0]:
                    if len(bucket) >= n_each or int(t) in used:
                        continue
                    used.add(int(t))
                    bucket.append((int(ci[t]), p[t].copy()))
    return reject, accept
