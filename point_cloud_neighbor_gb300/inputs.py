"""Seeded synthetic point clouds for the five benchmark workloads.

This module is the only code that both the oracle side and the CUDA side of
the tests (and the benchmark) share.  It draws coordinates and nothing else:
no squared distance, threshold, selection or ordering rule of FPS / kNN /
Ball Query is computed here.  Everything is generated with numpy's
``default_rng`` (PCG64) in float64 and rounded once to float32, so that the
oracle and the GPU read identical bytes.

The shapes follow the workloads the mps-pointops project page benchmarks on
("Benchmark": random-order 100k-point clouds near a sphere at MulSen-AD
scale; "Real data: MulSen-AD grouping": Point-MAE Group(1024, 128)), restated
synthetically:

====  ======================================================================
cfg   construction
====  ======================================================================
1     Tiny: B=1, N=1024 uniform in [0,1)^3 snapped to the 1/64 grid, then 32
      randomly chosen points overwritten by copies of 32 others (exact ties).
2     Point-MAE grouping: B=32 clouds of N=8192 points, uniform on the unit
      sphere (normalised normals) plus N(0, 0.01^2) jitter per coordinate.
3     PointNet++ set abstraction: B=16, N=4096 uniform in [-1,1)^3.
4     Single large cloud: B=1, N=100,000 from a mixture of 64 isotropic
      Gaussians (sigma=0.05, means uniform in [0,1)^3, equal weights),
      shuffled; ``morton=True`` gives the same points Morton-sorted.
5     Very large cloud: B=1, N=1,000,000 uniform in [0,1)^3 with 10,000
      points overwritten by copies of other points (1% exact duplicates).
====  ======================================================================
"""
from __future__ import annotations

import numpy as np

# Operator parameters of each workload (not computed, only stated).
CONFIGS = {
    "tiny": dict(seed=0, B=1, N=1024, npoint=64, start_idx=0, knn_k=16,
                 bq=[(0.125, 16)]),
    "point_mae": dict(seed=1, B=32, N=8192, npoint=512, start_idx=0,
                      knn_k=32, bq=[]),
    "pointnet2": dict(seed=2, B=16, N=4096, npoint=1024, start_idx=0,
                      knn_k=3, bq=[(0.1, 32), (0.2, 64)]),
    "large": dict(seed=3, B=1, N=100_000, npoint=4096, start_idx=0,
                  knn_k=16, bq=[(0.02, 32)]),
    "very_large": dict(seed=4, B=1, N=1_000_000, npoint=16384, start_idx=0,
                       knn_k=32, bq=[(0.01, 64)]),
}


def uniform(rng: np.random.Generator, B: int, N: int, lo: float = 0.0,
            hi: float = 1.0) -> np.ndarray:
    """[B,N,3] float32 uniform in [lo, hi)^3."""
    return (lo + (hi - lo) * rng.random((B, N, 3))).astype(np.float32)


def tiny(seed: int = 0, N: int = 1024, n_dup: int = 32) -> np.ndarray:
    """Workload 1: [1,N,3], coordinates on the 1/64 grid, n_dup exact copies."""
    rng = np.random.default_rng(seed)
    u = rng.random((N, 3))
    x = np.floor(u * 64.0) / 64.0
    perm = rng.permutation(N)
    dst, src = perm[:n_dup], perm[n_dup:2 * n_dup]
    x[dst] = x[src]
    return x.astype(np.float32)[None]


def point_mae(seed: int = 1, B: int = 32, N: int = 8192,
              jitter: float = 0.01) -> np.ndarray:
    """Workload 2: [B,N,3] points on the unit sphere plus Gaussian jitter."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((B, N, 3))
    v /= np.linalg.norm(v, axis=-1, keepdims=True)
    v += jitter * rng.standard_normal((B, N, 3))
    return v.astype(np.float32)


def pointnet2(seed: int = 2, B: int = 16, N: int = 4096) -> np.ndarray:
    """Workload 3: [B,N,3] uniform in [-1,1)^3."""
    return uniform(np.random.default_rng(seed), B, N, -1.0, 1.0)


def morton_order(x: np.ndarray, bits: int = 10) -> np.ndarray:
    """Permutation sorting one cloud [N,3] by its Morton (Z-order) code.

    Each axis is quantised to ``bits`` bits over the cloud's bounding box and
    the bits are interleaved (x lowest).  The sort is stable, so equal codes
    keep their original order.
    """
    x = np.asarray(x, dtype=np.float64)
    lo = x.min(axis=0)
    span = np.maximum(x.max(axis=0) - lo, 1e-300)
    q = np.floor((x - lo) / span * (1 << bits)).astype(np.int64)
    q = np.clip(q, 0, (1 << bits) - 1)
    code = np.zeros(x.shape[0], dtype=np.int64)
    for bit in range(bits):
        for axis in range(3):
            code |= ((q[:, axis] >> bit) & 1) << (3 * bit + axis)
    return np.argsort(code, kind="stable")


def large(seed: int = 3, N: int = 100_000, n_clusters: int = 64,
          sigma: float = 0.05, morton: bool = False) -> np.ndarray:
    """Workload 4: [1,N,3] Gaussian mixture, random order or Morton-sorted."""
    rng = np.random.default_rng(seed)
    means = rng.random((n_clusters, 3))
    label = rng.integers(0, n_clusters, size=N)
    x = means[label] + sigma * rng.standard_normal((N, 3))
    x = x[rng.permutation(N)].astype(np.float32)
    if morton:
        x = x[morton_order(x)]
    return np.ascontiguousarray(x)[None]


def very_large(seed: int = 4, N: int = 1_000_000,
               n_dup: int = 10_000) -> np.ndarray:
    """Workload 5: [1,N,3] uniform in [0,1)^3 with n_dup exact duplicates."""
    rng = np.random.default_rng(seed)
    x = rng.random((N, 3))
    perm = rng.permutation(N)
    dst, src = perm[:n_dup], perm[n_dup:2 * n_dup]
    x[dst] = x[src]
    return x.astype(np.float32)[None]


def make(name: str, **kw) -> np.ndarray:
    """The point cloud of the named workload (see CONFIGS)."""
    fn = {"tiny": tiny, "point_mae": point_mae, "pointnet2": pointnet2,
          "large": large, "very_large": very_large}[name]
    return fn(**kw)


def random_cloud(seed: int, B: int, N: int, lo: float = -1.0,
                 hi: float = 1.0, grid: float | None = None) -> np.ndarray:
    """Small random clouds for edge-case tests; optional snapping to a grid."""
    rng = np.random.default_rng(seed)
    x = lo + (hi - lo) * rng.random((B, N, 3))
    if grid is not None:
        x = np.floor(x / grid) * grid
    return x.astype(np.float32)


def sample_rows(seed: int, total: int, n: int) -> np.ndarray:
    """n distinct flat query rows out of ``total``, sorted (for sampled checks)."""
    rng = np.random.default_rng(seed)
    n = min(n, total)
    return np.sort(rng.choice(total, size=n, replace=False)).astype(np.int64)
