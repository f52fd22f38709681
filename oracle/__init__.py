"""The oracle: a plain, slow CPU statement of FPS, kNN and Ball Query.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``point_cloud_neighbor_gb300``) never imports, loads or calls it, and it
imports nothing from the product path.

The arithmetic lives in ``pc_oracle.c`` (float32, one rounding per operation,
compiled with ``-ffp-contract=off``), which follows the mps-pointops 0.5.0
project page, "The operators in equations", and the "Numerical contracts"
page, "Selection and output".  This module only builds that file with gcc,
loads it with ctypes and marshals numpy arrays.  Rows of independent queries
(and clouds for FPS) can be spread over host threads: ctypes releases the GIL
during each call, and every row is computed by the same plain C loop.

Pins (what ties this oracle to something other than itself) are in
``tests/test_oracle_pins.py``; the readings of the pages it takes are listed
in the repository's design notes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpc_oracle.so")

# -ffp-contract=off: no a*b+c -> fma contraction (GCC on aarch64 contracts by
# default).  No -ffast-math, no -ffinite-math-only: IEEE semantics, subnormals
# kept.  -fno-builtin-sqrtf is not needed: sqrtf is correctly rounded anyway.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared"]

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``pc_oracle.c`` into ``oracle/_build/libpc_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int64
    lib.orc_s32.restype = ctypes.c_float
    lib.orc_s32.argtypes = [P, P]
    lib.orc_radius_threshold.restype = ctypes.c_float
    lib.orc_radius_threshold.argtypes = [ctypes.c_double]
    lib.orc_fps.restype = ctypes.c_int
    lib.orc_fps.argtypes = [P, I, I, I, I, P]
    lib.orc_fps_threads.restype = ctypes.c_int
    lib.orc_fps_threads.argtypes = [P, I, I, I, I, I, P]
    lib.orc_min_dist_to_set.restype = ctypes.c_int
    lib.orc_min_dist_to_set.argtypes = [P, I, P, I, P, I, P]
    lib.orc_knn_rows.restype = ctypes.c_int
    lib.orc_knn_rows.argtypes = [P, I, I, P, I, I, P, I, P, P]
    lib.orc_ball_query_rows.restype = ctypes.c_int
    lib.orc_ball_query_rows.argtypes = [P, I, I, P, I, ctypes.c_double,
                                        I, P, I, P, P]
    lib.orc_ball_query_scan_len.restype = ctypes.c_int
    lib.orc_ball_query_scan_len.argtypes = [P, I, I, P, I,
                                            ctypes.c_double, I, P, I, P]
    lib.orc_s32_pairs.restype = None
    lib.orc_s32_pairs.argtypes = [P, P, I, P]
    lib.orc_sd.restype = ctypes.c_float
    lib.orc_sd.argtypes = [P, P, I]
    lib.orc_knn_d_rows.restype = ctypes.c_int
    lib.orc_knn_d_rows.argtypes = [P, I, I, P, I, I, I, ctypes.c_int, P, I, P, P]
    lib.orc_knn_masked_rows.restype = ctypes.c_int
    lib.orc_knn_masked_rows.argtypes = [P, I, I, P, I, I, P, P, ctypes.c_int,
                                        P, I, P, P]
    lib.orc_ball_query_masked_rows.restype = ctypes.c_int
    lib.orc_ball_query_masked_rows.argtypes = [P, I, I, P, I, P, P,
                                               ctypes.c_double, I, P, I, P, P]
    lib.orc_gather_points.restype = ctypes.c_int
    lib.orc_gather_points.argtypes = [P, I, I, P, I, I, P]
    lib.orc_three_interpolate.restype = ctypes.c_int
    lib.orc_three_interpolate.argtypes = [P, I, I, I, P, P, I, P]
    lib.orc_three_interpolate_backward.restype = ctypes.c_int
    lib.orc_three_interpolate_backward.argtypes = [P, I, I, I, P, P, I, P]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (used by the tests that
    plant a mistake in the oracle to show that the pins catch it)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", *CFLAGS, src, "-o", out_path, "-lm", "-lpthread"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


class use_library:
    """Context manager: route this module's calls to another build of the
    oracle source (a planted-mistake variant) for the duration."""

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self.saved = _lib
            _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _split(n: int, parts: int):
    if n <= 0:
        return []
    parts = max(1, min(parts, n))
    step = -(-n // parts)
    return [(i, min(n, i + step)) for i in range(0, n, step)]


def s32(a, b) -> np.ndarray:
    """Squared distances s32(a_i, b_i) of matching rows of two [n,3] arrays."""
    a = _f32(a).reshape(-1, 3)
    b = _f32(b).reshape(-1, 3)
    assert a.shape == b.shape
    out = np.empty(a.shape[0], dtype=np.float32)
    _load().orc_s32_pairs(_ptr(a), _ptr(b), a.shape[0], _ptr(out))
    return out


def radius_threshold(radius: float) -> np.float32:
    """R2 = fl32(fl32(r) * fl32(r))."""
    return np.float32(_load().orc_radius_threshold(float(radius)))


def fps(xyz, npoint: int, start_idx: int = 0, threads: int = 1) -> np.ndarray:
    """Farthest point sampling of every cloud of ``xyz`` [B,N,3] -> [B,npoint]."""
    xyz = _f32(xyz)
    B, N, _ = xyz.shape
    out = np.empty((B, npoint), dtype=np.int64)
    lib = _load()

    def run(lo, hi):
        if hi <= lo:
            return
        sub = np.ascontiguousarray(xyz[lo:hi])
        o = np.empty((hi - lo, npoint), dtype=np.int64)
        _check(lib.orc_fps(_ptr(sub), hi - lo, N, npoint, start_idx, _ptr(o)),
               "fps")
        out[lo:hi] = o

    chunks = _split(B, threads)
    if len(chunks) <= 1:
        run(0, B)
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(lambda c: run(*c), chunks))
    return out


def fps_all_cores(xyz, npoint: int, start_idx: int = 0,
                  threads: int | None = None) -> np.ndarray:
    """Farthest point sampling with each step's points split over host
    threads (one cloud after another): the all-core CPU baseline.  Returns
    what ``fps`` returns; the tests check the two are equal."""
    xyz = _f32(xyz)
    B, N, _ = xyz.shape
    threads = default_threads() if threads is None else int(threads)
    out = np.empty((B, npoint), dtype=np.int64)
    _check(_load().orc_fps_threads(_ptr(xyz), B, N, npoint, start_idx,
                                   max(1, threads), _ptr(out)), "fps_all_cores")
    return out


def min_dist_to_set(x, centers, points) -> np.ndarray:
    """m_j = min_u s32(x_j, x_{centers[u]}) for each j in ``points`` (one cloud)."""
    x = _f32(x).reshape(-1, 3)
    centers = np.ascontiguousarray(centers, dtype=np.int64)
    points = np.ascontiguousarray(points, dtype=np.int64)
    out = np.empty(points.shape[0], dtype=np.float32)
    _check(_load().orc_min_dist_to_set(_ptr(x), x.shape[0], _ptr(centers),
                                       centers.shape[0], _ptr(points),
                                       points.shape[0], _ptr(out)),
           "min_dist_to_set")
    return out


def _rows_arg(rows, total):
    if rows is None:
        return np.arange(total, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def knn(query, ref, k: int, rows=None, threads: int = 1):
    """kNN of query [B,Q,3] against ref [B,N,3].

    Returns (dist [R,k] float32, idx [R,k] int64) for the flat rows ``rows``
    (row = b*Q + i; all B*Q rows when ``rows`` is None).
    """
    query = _f32(query)
    ref = _f32(ref)
    B, Q, _ = query.shape
    N = ref.shape[1]
    rows = _rows_arg(rows, B * Q)
    R = rows.shape[0]
    dist = np.empty((R, k), dtype=np.float32)
    idx = np.empty((R, k), dtype=np.int64)
    lib = _load()

    def run(lo, hi):
        if hi <= lo:
            return
        rr = np.ascontiguousarray(rows[lo:hi])
        d = np.empty((hi - lo, k), dtype=np.float32)
        i = np.empty((hi - lo, k), dtype=np.int64)
        _check(lib.orc_knn_rows(_ptr(query), B, Q, _ptr(ref), N, k, _ptr(rr),
                                hi - lo, _ptr(d), _ptr(i)), "knn")
        dist[lo:hi] = d
        idx[lo:hi] = i

    chunks = _split(R, threads)
    if len(chunks) <= 1:
        run(0, R)
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(lambda c: run(*c), chunks))
    return dist, idx


def ball_query(query, ref, radius: float, K: int, rows=None, threads: int = 1):
    """First-K Ball Query of query [B,Q,3] against ref [B,N,3].

    Returns (dist2 [R,K] float32, idx [R,K] int64) for the flat rows ``rows``.
    """
    query = _f32(query)
    ref = _f32(ref)
    B, Q, _ = query.shape
    N = ref.shape[1]
    rows = _rows_arg(rows, B * Q)
    R = rows.shape[0]
    dist2 = np.empty((R, K), dtype=np.float32)
    idx = np.empty((R, K), dtype=np.int64)
    lib = _load()

    def run(lo, hi):
        if hi <= lo:
            return
        rr = np.ascontiguousarray(rows[lo:hi])
        d = np.empty((hi - lo, K), dtype=np.float32)
        i = np.empty((hi - lo, K), dtype=np.int64)
        _check(lib.orc_ball_query_rows(_ptr(query), B, Q, _ptr(ref), N,
                                       float(radius), K, _ptr(rr), hi - lo,
                                       _ptr(d), _ptr(i)), "ball_query")
        dist2[lo:hi] = d
        idx[lo:hi] = i

    chunks = _split(R, threads)
    if len(chunks) <= 1:
        run(0, R)
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(lambda c: run(*c), chunks))
    return dist2, idx


def ball_query_scan_len(query, ref, radius: float, K: int, rows=None,
                        threads: int = 1) -> np.ndarray:
    """Pairs the first-K rule must examine per row (position of K-th hit + 1, or N)."""
    query = _f32(query)
    ref = _f32(ref)
    B, Q, _ = query.shape
    N = ref.shape[1]
    rows = _rows_arg(rows, B * Q)
    R = rows.shape[0]
    out = np.empty(R, dtype=np.int64)
    lib = _load()

    def run(lo, hi):
        if hi <= lo:
            return
        rr = np.ascontiguousarray(rows[lo:hi])
        o = np.empty(hi - lo, dtype=np.int64)
        _check(lib.orc_ball_query_scan_len(_ptr(query), B, Q, _ptr(ref), N,
                                           float(radius), K, _ptr(rr),
                                           hi - lo, _ptr(o)), "scan_len")
        out[lo:hi] = o

    chunks = _split(R, threads)
    if len(chunks) <= 1:
        run(0, R)
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(lambda c: run(*c), chunks))
    return out


# ---------------------------------------------------------------------------
# Lengths-masked kNN / Ball Query, gather, three_interpolate, Chamfer.
# ---------------------------------------------------------------------------
def _lens(lengths, B):
    if lengths is None:
        return None
    a = np.ascontiguousarray(lengths, dtype=np.int64)
    if a.shape != (B,):
        raise ValueError(f"lengths must have shape [{B}]")
    return a


def _opt_ptr(a):
    return None if a is None else _ptr(a)


def knn_masked(query, ref, k: int, query_lengths=None, ref_lengths=None,
               squared: bool = False, rows=None, threads: int = 1):
    """kNN over the valid prefix of every cloud (``orc_knn_masked_rows``).

    Returns (dist [R,k], idx [R,k]); dist is s when ``squared`` else sqrt(s);
    rows past the query length and slots past the references are (0, -1).
    """
    query = _f32(query)
    ref = _f32(ref)
    B, Q, _ = query.shape
    N = ref.shape[1]
    ql, rl = _lens(query_lengths, B), _lens(ref_lengths, B)
    rows = _rows_arg(rows, B * Q)
    R = rows.shape[0]
    dist = np.empty((R, k), dtype=np.float32)
    idx = np.empty((R, k), dtype=np.int64)
    lib = _load()

    def run(lo, hi):
        if hi <= lo:
            return
        rr = np.ascontiguousarray(rows[lo:hi])
        d = np.empty((hi - lo, k), dtype=np.float32)
        i = np.empty((hi - lo, k), dtype=np.int64)
        _check(lib.orc_knn_masked_rows(_ptr(query), B, Q, _ptr(ref), N, k,
                                       _opt_ptr(ql), _opt_ptr(rl), int(squared),
                                       _ptr(rr), hi - lo, _ptr(d), _ptr(i)),
               "knn_masked")
        dist[lo:hi] = d
        idx[lo:hi] = i

    chunks = _split(R, threads)
    if len(chunks) <= 1:
        run(0, R)
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(lambda c: run(*c), chunks))
    return dist, idx


def ball_query_masked(query, ref, radius: float, K: int, query_lengths=None,
                      ref_lengths=None, rows=None):
    """First-K Ball Query over the valid prefix of every cloud."""
    query = _f32(query)
    ref = _f32(ref)
    B, Q, _ = query.shape
    N = ref.shape[1]
    ql, rl = _lens(query_lengths, B), _lens(ref_lengths, B)
    rows = _rows_arg(rows, B * Q)
    R = rows.shape[0]
    d = np.empty((R, K), dtype=np.float32)
    i = np.empty((R, K), dtype=np.int64)
    _check(_load().orc_ball_query_masked_rows(
        _ptr(query), B, Q, _ptr(ref), N, _opt_ptr(ql), _opt_ptr(rl),
        float(radius), K, _ptr(rows), R, _ptr(d), _ptr(i)), "ball_query_masked")
    return d, i


def gather_points(x, idx) -> np.ndarray:
    """out[b,i,t,:] = x[b, idx[b,i,t], :], zeros where idx = -1."""
    x = _f32(x)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    B, N, _ = x.shape
    _, Q, K = idx.shape
    out = np.empty((B, Q, K, 3), dtype=np.float32)
    _check(_load().orc_gather_points(_ptr(x), B, N, _ptr(idx), Q, K, _ptr(out)),
           "gather_points")
    return out


def three_interpolate(features, idx, weight) -> np.ndarray:
    """features [B,C,M], idx [B,n,3] int64, weight [B,n,3] -> [B,C,n]."""
    f = np.ascontiguousarray(features, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    w = np.ascontiguousarray(weight, dtype=np.float32)
    B, C, M = f.shape
    n = idx.shape[1]
    out = np.empty((B, C, n), dtype=np.float32)
    _check(_load().orc_three_interpolate(_ptr(f), B, C, M, _ptr(idx), _ptr(w),
                                         n, _ptr(out)), "three_interpolate")
    return out


def three_interpolate_backward(grad_out, idx, weight, M: int) -> np.ndarray:
    """grad_out [B,C,n] -> grad_features [B,C,M] (sequential float32 sums)."""
    g = np.ascontiguousarray(grad_out, dtype=np.float32)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    w = np.ascontiguousarray(weight, dtype=np.float32)
    B, C, n = g.shape
    out = np.empty((B, C, M), dtype=np.float32)
    _check(_load().orc_three_interpolate_backward(_ptr(g), B, C, n, _ptr(idx),
                                                  _ptr(w), M, _ptr(out)),
           "three_interpolate_backward")
    return out


REDUCTIONS = ("none", "sum", "mean")


def chamfer(x, y, x_lengths=None, y_lengths=None, weights=None,
            point_reduction: str = "mean", batch_reduction: str = "mean",
            single_directional: bool = False, threads: int = 1):
    """Bidirectional squared-L2 Chamfer distance (project page, "Roadmap",
    Phase 4):  L = sum_i |q_i - x_a(i)|^2 + sum_j |x_j - q_b(j)|^2, with a(i)
    the nearest point of y to x_i and b(j) the nearest point of x to y_j
    (kNN with k = 1: smallest (s, index)).

    Readings taken (the pages name lengths, weights, point and batch
    reductions without giving their divisors): points past a cloud's length
    are excluded as queries and as references; a point with no valid
    reference contributes 0 and gets index -1; "mean" over points divides a
    cloud's sum by max(length, 1); weights [B] scale each cloud's loss;
    "mean" over the batch divides by B.  Sums are exact (math.fsum over the
    float32 terms), the divisions and products are in float64, and the
    result is rounded once to float32.

    Returns (loss, (dist_x [B,P1], idx_x [B,P1]), (dist_y, idx_y) or None):
    loss is a float32 scalar, or [B] float32 for batch_reduction "none".
    """
    import math
    x = _f32(x)
    y = _f32(y)
    B, P1, _ = x.shape
    P2 = y.shape[1]
    xl, yl = _lens(x_lengths, B), _lens(y_lengths, B)
    dx, ix = knn_masked(x, y, 1, xl, yl, squared=True, threads=threads)
    dx, ix = dx.reshape(B, P1), ix.reshape(B, P1)
    if single_directional:
        dy = iy = None
    else:
        dy, iy = knn_masked(y, x, 1, yl, xl, squared=True, threads=threads)
        dy, iy = dy.reshape(B, P2), iy.reshape(B, P2)
    if point_reduction not in ("sum", "mean") or batch_reduction not in REDUCTIONS:
        raise ValueError("point_reduction: sum|mean; batch_reduction: none|sum|mean")

    def clamp(lens, b, full):
        if lens is None:
            return full
        return min(max(int(lens[b]), 0), full)

    per = []
    for b in range(B):
        nx = clamp(xl, b, P1)
        t = math.fsum(float(v) for v in dx[b, :nx])
        if point_reduction == "mean":
            t = t / max(nx, 1)
        if not single_directional:
            ny = clamp(yl, b, P2)
            u = math.fsum(float(v) for v in dy[b, :ny])
            if point_reduction == "mean":
                u = u / max(ny, 1)
            t = t + u
        if weights is not None:
            t = t * float(np.float32(weights[b]))
        per.append(t)
    if batch_reduction == "none":
        loss = np.array(per, dtype=np.float64).astype(np.float32)
    elif batch_reduction == "sum":
        loss = np.float32(math.fsum(per))
    else:
        loss = np.float32(math.fsum(per) / B) if B > 0 else np.float32(0.0)
    return loss, (dx, ix), (None if single_directional else (dy, iy))


def sd(a, b) -> np.float32:
    """Dimension-by-dimension squared distance of two float32 vectors."""
    a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    b = np.ascontiguousarray(b, dtype=np.float32).reshape(-1)
    return np.float32(_load().orc_sd(_ptr(a), _ptr(b), a.shape[0]))


def knn_d(query, ref, k: int, squared: bool = False, rows=None, threads: int = 1):
    """kNN of query [B,Q,D] against ref [B,N,D] with the dimension-by-dimension
    distance (``orc_knn_d_rows``); returns (dist [R,k], idx [R,k])."""
    query = np.ascontiguousarray(query, dtype=np.float32)
    ref = np.ascontiguousarray(ref, dtype=np.float32)
    B, Q, D = query.shape
    N = ref.shape[1]
    if ref.shape[2] != D:
        raise ValueError("query and ref dimensions differ")
    rows = _rows_arg(rows, B * Q)
    R = rows.shape[0]
    dist = np.empty((R, k), dtype=np.float32)
    idx = np.empty((R, k), dtype=np.int64)
    lib = _load()

    def run(lo, hi):
        if hi <= lo:
            return
        rr = np.ascontiguousarray(rows[lo:hi])
        d = np.empty((hi - lo, k), dtype=np.float32)
        i = np.empty((hi - lo, k), dtype=np.int64)
        _check(lib.orc_knn_d_rows(_ptr(query), B, Q, _ptr(ref), N, D, k,
                                  int(squared), _ptr(rr), hi - lo, _ptr(d),
                                  _ptr(i)), "knn_d")
        dist[lo:hi] = d
        idx[lo:hi] = i

    chunks = _split(R, threads)
    if len(chunks) <= 1:
        run(0, R)
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            list(ex.map(lambda c: run(*c), chunks))
    return dist, idx
