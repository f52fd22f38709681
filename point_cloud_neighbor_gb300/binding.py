"""Thin Python binding of libpointcloud.so (include/pointcloud.h).

Argument marshalling only: the functions check tensor placement, dtype,
layout and shapes, allocate outputs with torch's caching allocator, pass raw
device pointers and the current CUDA stream through ctypes, and turn a
non-OK status into :class:`PointCloudError`.  Every step of FPS, kNN and Ball
Query runs in the library's CUDA kernels.  There is no CPU path: CPU
tensors, a missing library or a non-sm_103 device raise.

Names follow the C ABI (``pc_fps``, ``pc_knn``, ``pc_ball_query``); the
aliases ``furthest_point_sample``, ``knn`` and ``ball_query`` mirror the
mps-pointops dense API ("Contracts" section of its project page).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpointcloud.so")

PC_OK = 0
PC_ERR_INVALID_ARGUMENT = 1
PC_ERR_UNSUPPORTED = 2
PC_ERR_CUDA = 3
PC_ERR_DEVICE_TIMEOUT = 4
PC_ERR_NO_DEVICE = 5

PC_FPS_AUTO, PC_FPS_BLOCK, PC_FPS_CLUSTER, PC_FPS_GRID = 0, 1, 2, 3
PC_KNN_SQUARED = 1
PC_REDUCTION_NONE, PC_REDUCTION_SUM, PC_REDUCTION_MEAN = 0, 1, 2

# Every symbol include/pointcloud.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int64
_SIGNATURES = {
    "pc_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pc_last_error_message": (ctypes.c_char_p, []),
    "pc_version": (ctypes.c_int, []),
    "pc_fps": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "pc_fps_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "pc_fps_ex": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P, ctypes.c_size_t,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]),
    "pc_fps_workspace_bytes_ex": (ctypes.c_size_t, [_I, _I, _I, ctypes.c_int,
                                                    ctypes.c_int]),
    "pc_fps_grid_static": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, ctypes.c_int,
                                          _P]),
    "pc_knn": (ctypes.c_int, [_P, _I, _I, _P, _I, _I, _P, _P, _P]),
    "pc_grid_bytes": (ctypes.c_size_t, [_I, _I]),
    "pc_grid_build": (ctypes.c_int, [_P, _I, _I, _P, ctypes.c_size_t, _P]),
    "pc_knn_grid": (ctypes.c_int, [_P, _I, _I, _P, _I, _I, _P, _P, _P]),
    "pc_ball_query_grid": (ctypes.c_int, [_P, _I, _I, _P, _I, ctypes.c_double,
                                          _I, _P, _P, _P]),
    "pc_ball_query": (ctypes.c_int, [_P, _I, _I, _P, _I, ctypes.c_double, _I,
                                     _P, _P, _P]),
    "pc_knn_ball_query": (ctypes.c_int, [_P, _I, _I, _P, _I, _I, _P, _P,
                                         ctypes.c_double, _I, _P, _P, _P]),
    "pc_knn_ball_query_plan": (ctypes.c_int, [_I, _I, _I, _I, ctypes.c_double,
                                              _I, ctypes.POINTER(ctypes.c_int)]),
    "pc_knn_ex": (ctypes.c_int, [_P, _I, _I, _P, _I, _I, _P, _P, ctypes.c_int,
                                 _P, _P, _P]),
    "pc_ball_query_ex": (ctypes.c_int, [_P, _I, _I, _P, _I, _P, _P,
                                        ctypes.c_double, _I, _P, _P, _P]),
    "pc_chamfer": (ctypes.c_int, [_P, _I, _I, _P, _I, _P, _P, _P, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, _P, _P, _P, _P,
                                  _P, _P]),
    "pc_three_interpolate": (ctypes.c_int, [_P, _I, _I, _I, _P, _P, _I, _P, _P]),
    "pc_three_interpolate_backward": (ctypes.c_int, [_P, _I, _I, _I, _P, _P, _I,
                                                     _P, _P]),
    "pc_gather_points": (ctypes.c_int, [_P, _I, _I, _P, _I, _I, _P, _P]),
    "pc_knn_d": (ctypes.c_int, [_P, _I, _I, _P, _I, _I, _I, ctypes.c_int, _P, _P,
                                _P]),
    "pc_device_status": (ctypes.c_int, [_P, ctypes.c_int,
                                        ctypes.POINTER(ctypes.c_int32)]),
    "pc_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "pc_debug_set_fps_grid_stall": (None, [ctypes.c_int]),
    "pc_debug_set_stall": (None, [ctypes.c_int]),
    "pc_set_sm_reserve": (None, [ctypes.c_int]),
    "pc_fps_set_batched": (ctypes.c_int, [ctypes.c_int]),
    "pc_fps_sm_count": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]),
    "pc_fps_plan": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_int),
                                   ctypes.POINTER(ctypes.c_int),
                                   ctypes.POINTER(ctypes.c_int)]),
}

_lib = None
_lock = threading.Lock()


class PointCloudError(RuntimeError):
    """A library call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libpointcloud.so (built by ``point_cloud_neighbor_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build the CUDA library first "
                    "(python -m point_cloud_neighbor_gb300.build); there is no "
                    "CPU fallback")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def exported_symbols():
    return list(_SIGNATURES)


def _raise_on(status: int, what: str):
    if status != PC_OK:
        L = lib()
        name = L.pc_status_string(status).decode()
        msg = L.pc_last_error_message().decode()
        raise PointCloudError(status, f"{what}: {name}: {msg}")


def _stream_ptr(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_cloud(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); "
                         "this library has no CPU path")
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32 (got {t.dtype})")
    if t.dim() != 3 or t.shape[-1] != 3:
        raise ValueError(f"{name} must have shape [B, N, 3] (got {tuple(t.shape)})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def pc_fps(xyz: torch.Tensor, npoint: int, start_idx: int = 0, *,
           strategy: int = PC_FPS_AUTO, cluster_size: int = 0,
           blocks_per_cloud: int = 0, out: torch.Tensor | None = None,
           workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Farthest point sampling: [B,N,3] float32 -> [B,npoint] int64."""
    _check_cloud(xyz, "xyz")
    B, N, _ = xyz.shape
    L = lib()
    with torch.cuda.device(xyz.device):
        if out is None:
            out = torch.empty((B, npoint), dtype=torch.int64, device=xyz.device)
        ws_ptr, ws_bytes = None, 0
        if B > 0 and N > 0 and cluster_size == 0:
            # (an explicit cluster size: the library sizes the scratch)
            need = L.pc_fps_workspace_bytes_ex(B, N, npoint, strategy,
                                               blocks_per_cloud)
            if need:
                if workspace is None or workspace.numel() < need:
                    workspace = torch.empty(need, dtype=torch.uint8,
                                            device=xyz.device)
                ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
        st = L.pc_fps_ex(xyz.data_ptr(), B, N, npoint, start_idx,
                         out.data_ptr(), ws_ptr, ws_bytes, strategy,
                         cluster_size, blocks_per_cloud,
                         _stream_ptr(xyz.device))
    _raise_on(st, "pc_fps")
    return out


def _check_lengths(t, B: int, device, name: str):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != torch.int64 or tuple(t.shape) != (B,) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int64 tensor of shape [{B}]")
    return t


def _ptr_or_none(t):
    return None if t is None else t.data_ptr()


def pc_knn(query: torch.Tensor, ref: torch.Tensor, k: int, *,
           query_lengths: torch.Tensor | None = None,
           ref_lengths: torch.Tensor | None = None, squared: bool = False,
           out_dist: torch.Tensor | None = None,
           out_idx: torch.Tensor | None = None):
    """k nearest neighbors: returns (dist [B,Q,k] float32, idx [B,Q,k] int64).

    With ``query_lengths`` / ``ref_lengths`` ([B] int64) or ``squared`` the
    call goes to pc_knn_ex: masked rows and missing neighbors are (0, -1), and
    ``squared`` returns s instead of sqrt(s).
    """
    _check_cloud(query, "query")
    _check_cloud(ref, "ref")
    B, Q, _ = query.shape
    if ref.shape[0] != B:
        raise ValueError("query and ref must have the same batch size")
    if ref.device != query.device:
        raise ValueError("query and ref must be on the same device")
    N = ref.shape[1]
    ql = _check_lengths(query_lengths, B, query.device, "query_lengths")
    rl = _check_lengths(ref_lengths, B, query.device, "ref_lengths")
    L = lib()
    with torch.cuda.device(query.device):
        if out_dist is None:
            out_dist = torch.empty((B, Q, k), dtype=torch.float32,
                                   device=query.device)
        if out_idx is None:
            out_idx = torch.empty((B, Q, k), dtype=torch.int64,
                                  device=query.device)
        if ql is None and rl is None and not squared:
            st = L.pc_knn(query.data_ptr(), B, Q, ref.data_ptr(), N, k,
                          out_dist.data_ptr(), out_idx.data_ptr(),
                          _stream_ptr(query.device))
        else:
            st = L.pc_knn_ex(query.data_ptr(), B, Q,
                             ref.data_ptr() if N > 0 else None, N, k,
                             _ptr_or_none(ql), _ptr_or_none(rl),
                             PC_KNN_SQUARED if squared else 0,
                             out_dist.data_ptr(), out_idx.data_ptr(),
                             _stream_ptr(query.device))
    _raise_on(st, "pc_knn")
    return out_dist, out_idx


def pc_ball_query(query: torch.Tensor, ref: torch.Tensor, radius: float,
                  K: int, *, query_lengths: torch.Tensor | None = None,
                  ref_lengths: torch.Tensor | None = None,
                  out_dist2: torch.Tensor | None = None,
                  out_idx: torch.Tensor | None = None):
    """First-K Ball Query: returns (dist2 [B,Q,K] float32, idx [B,Q,K] int64).

    With ``query_lengths`` / ``ref_lengths`` ([B] int64) the call goes to
    pc_ball_query_ex (rows past a cloud's query length are padding).
    """
    _check_cloud(query, "query")
    _check_cloud(ref, "ref")
    B, Q, _ = query.shape
    if ref.shape[0] != B:
        raise ValueError("query and ref must have the same batch size")
    if ref.device != query.device:
        raise ValueError("query and ref must be on the same device")
    N = ref.shape[1]
    ql = _check_lengths(query_lengths, B, query.device, "query_lengths")
    rl = _check_lengths(ref_lengths, B, query.device, "ref_lengths")
    L = lib()
    with torch.cuda.device(query.device):
        if out_dist2 is None:
            out_dist2 = torch.empty((B, Q, K), dtype=torch.float32,
                                    device=query.device)
        if out_idx is None:
            out_idx = torch.empty((B, Q, K), dtype=torch.int64,
                                  device=query.device)
        if ql is None and rl is None:
            st = L.pc_ball_query(query.data_ptr(), B, Q,
                                 ref.data_ptr() if N > 0 else None, N,
                                 float(radius), K, out_dist2.data_ptr(),
                                 out_idx.data_ptr(), _stream_ptr(query.device))
        else:
            st = L.pc_ball_query_ex(query.data_ptr(), B, Q,
                                    ref.data_ptr() if N > 0 else None, N,
                                    _ptr_or_none(ql), _ptr_or_none(rl),
                                    float(radius), K, out_dist2.data_ptr(),
                                    out_idx.data_ptr(), _stream_ptr(query.device))
    _raise_on(st, "pc_ball_query")
    return out_dist2, out_idx


def pc_knn_ball_query(query: torch.Tensor, ref: torch.Tensor, k: int,
                      radius: float, K: int, *,
                      out: tuple | None = None):
    """kNN and first-K Ball Query of the same queries against the same
    references in one call: returns (knn_dist [B,Q,k], knn_idx [B,Q,k],
    bq_dist2 [B,Q,K], bq_idx [B,Q,K]), identical to :func:`pc_knn` and
    :func:`pc_ball_query`.  ``out`` may hold those four tensors."""
    _check_cloud(query, "query")
    _check_cloud(ref, "ref")
    B, Q, _ = query.shape
    if ref.shape[0] != B:
        raise ValueError("query and ref must have the same batch size")
    if ref.device != query.device:
        raise ValueError("query and ref must be on the same device")
    N = ref.shape[1]
    L = lib()
    with torch.cuda.device(query.device):
        if out is None:
            dev = query.device
            out = (torch.empty((B, Q, k), dtype=torch.float32, device=dev),
                   torch.empty((B, Q, k), dtype=torch.int64, device=dev),
                   torch.empty((B, Q, K), dtype=torch.float32, device=dev),
                   torch.empty((B, Q, K), dtype=torch.int64, device=dev))
        kd, ki, bd, bi = out
        for t, shape, dt, name in ((kd, (B, Q, k), torch.float32, "knn_dist"),
                                   (ki, (B, Q, k), torch.int64, "knn_idx"),
                                   (bd, (B, Q, K), torch.float32, "bq_dist2"),
                                   (bi, (B, Q, K), torch.int64, "bq_idx")):
            if (tuple(t.shape) != shape or t.dtype != dt or
                    t.device != query.device or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous {dt} tensor of "
                                 f"shape {shape} on {query.device}")
        st = L.pc_knn_ball_query(query.data_ptr(), B, Q,
                                 ref.data_ptr() if N > 0 else None, N, k,
                                 kd.data_ptr(), ki.data_ptr(), float(radius), K,
                                 bd.data_ptr(), bi.data_ptr(),
                                 _stream_ptr(query.device))
    _raise_on(st, "pc_knn_ball_query")
    return kd, ki, bd, bi


def pc_knn_ball_query_plan(B: int, Q: int, N: int, k: int, radius: float,
                           K: int) -> bool:
    """Whether :func:`pc_knn_ball_query` runs its fused pass for these sizes
    on the current device."""
    fused = ctypes.c_int(0)
    st = lib().pc_knn_ball_query_plan(B, Q, N, k, float(radius), K,
                                      ctypes.byref(fused))
    _raise_on(st, "pc_knn_ball_query_plan")
    return bool(fused.value)


class PointGrid:
    """A uniform grid over a reference cloud [B, N, 3] on the GPU (device
    memory owned by a torch tensor), for pc_knn_grid / pc_ball_query_grid."""

    def __init__(self, ref: torch.Tensor):
        _check_cloud(ref, "ref")
        self.B, self.N, _ = ref.shape
        self.device = ref.device
        L = lib()
        nbytes = L.pc_grid_bytes(self.B, self.N)
        self.buffer = torch.empty(max(nbytes, 256), dtype=torch.uint8,
                                  device=ref.device)
        with torch.cuda.device(ref.device):
            st = L.pc_grid_build(ref.data_ptr() if self.N > 0 else None,
                                 self.B, self.N, self.buffer.data_ptr(),
                                 self.buffer.numel(), _stream_ptr(ref.device))
        _raise_on(st, "pc_grid_build")


def pc_grid_build(ref: torch.Tensor) -> PointGrid:
    """Build the grid of reference cloud(s) ref [B, N, 3] float32 (CUDA)."""
    return PointGrid(ref)


def pc_knn_grid(query: torch.Tensor, grid: PointGrid, k: int, *,
                out_dist: torch.Tensor | None = None,
                out_idx: torch.Tensor | None = None):
    """kNN from a grid; same results as pc_knn(query, ref, k)."""
    _check_cloud(query, "query")
    B, Q, _ = query.shape
    if B != grid.B or query.device != grid.device:
        raise ValueError("query and grid must share batch size and device")
    L = lib()
    with torch.cuda.device(query.device):
        if out_dist is None:
            out_dist = torch.empty((B, Q, k), dtype=torch.float32, device=query.device)
        if out_idx is None:
            out_idx = torch.empty((B, Q, k), dtype=torch.int64, device=query.device)
        st = L.pc_knn_grid(query.data_ptr(), B, Q, grid.buffer.data_ptr(),
                           grid.N, k, out_dist.data_ptr(), out_idx.data_ptr(),
                           _stream_ptr(query.device))
    _raise_on(st, "pc_knn_grid")
    return out_dist, out_idx


def pc_ball_query_grid(query: torch.Tensor, grid: PointGrid, radius: float,
                       K: int, *, out_dist2: torch.Tensor | None = None,
                       out_idx: torch.Tensor | None = None):
    """Ball Query from a grid; same results as pc_ball_query(query, ref, r, K)."""
    _check_cloud(query, "query")
    B, Q, _ = query.shape
    if B != grid.B or query.device != grid.device:
        raise ValueError("query and grid must share batch size and device")
    L = lib()
    with torch.cuda.device(query.device):
        if out_dist2 is None:
            out_dist2 = torch.empty((B, Q, K), dtype=torch.float32, device=query.device)
        if out_idx is None:
            out_idx = torch.empty((B, Q, K), dtype=torch.int64, device=query.device)
        st = L.pc_ball_query_grid(query.data_ptr(), B, Q, grid.buffer.data_ptr(),
                                  grid.N, float(radius), K, out_dist2.data_ptr(),
                                  out_idx.data_ptr(), _stream_ptr(query.device))
    _raise_on(st, "pc_ball_query_grid")
    return out_dist2, out_idx


def pc_knn_d(query: torch.Tensor, ref: torch.Tensor, k: int, *,
             squared: bool = False, out_dist: torch.Tensor | None = None,
             out_idx: torch.Tensor | None = None):
    """kNN in D dimensions: query [B,Q,D], ref [B,N,D] float32 (CUDA) ->
    (dist [B,Q,k], idx [B,Q,k]); dimension-by-dimension accumulation."""
    for t, name in ((query, "query"), (ref, "ref")):
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor; this library has no CPU path")
        if t.dtype != torch.float32 or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor [B, n, D]")
    B, Q, D = query.shape
    if ref.shape[0] != B or ref.shape[2] != D or ref.device != query.device:
        raise ValueError("query and ref must share batch size, dimension and device")
    N = ref.shape[1]
    with torch.cuda.device(query.device):
        if out_dist is None:
            out_dist = torch.empty((B, Q, k), dtype=torch.float32, device=query.device)
        if out_idx is None:
            out_idx = torch.empty((B, Q, k), dtype=torch.int64, device=query.device)
        st = lib().pc_knn_d(query.data_ptr(), B, Q, ref.data_ptr(), N, D, k,
                            PC_KNN_SQUARED if squared else 0, out_dist.data_ptr(),
                            out_idx.data_ptr(), _stream_ptr(query.device))
    _raise_on(st, "pc_knn_d")
    return out_dist, out_idx


_REDUCTIONS = {"none": PC_REDUCTION_NONE, None: PC_REDUCTION_NONE,
               "sum": PC_REDUCTION_SUM, "mean": PC_REDUCTION_MEAN}


def pc_chamfer(x: torch.Tensor, y: torch.Tensor, *,
               x_lengths: torch.Tensor | None = None,
               y_lengths: torch.Tensor | None = None,
               weights: torch.Tensor | None = None,
               point_reduction: str = "mean", batch_reduction: str | None = "mean",
               single_directional: bool = False):
    """Squared-L2 Chamfer distance (forward).

    Returns (loss, (dist_x [B,P1], idx_x [B,P1]), (dist_y, idx_y) or None);
    loss is a 0-d float32 tensor, or [B] for batch_reduction "none"/None.
    """
    _check_cloud(x, "x")
    _check_cloud(y, "y")
    B, P1, _ = x.shape
    P2 = y.shape[1]
    if y.shape[0] != B or y.device != x.device:
        raise ValueError("x and y must share batch size and device")
    if point_reduction not in ("sum", "mean"):
        raise ValueError("point_reduction must be 'sum' or 'mean'")
    if batch_reduction not in _REDUCTIONS:
        raise ValueError("batch_reduction must be None, 'none', 'sum' or 'mean'")
    xl = _check_lengths(x_lengths, B, x.device, "x_lengths")
    yl = _check_lengths(y_lengths, B, x.device, "y_lengths")
    if weights is not None:
        if (not isinstance(weights, torch.Tensor) or weights.device != x.device
                or weights.dtype != torch.float32 or tuple(weights.shape) != (B,)
                or not weights.is_contiguous()):
            raise ValueError(f"weights must be a contiguous float32 CUDA tensor [{B}]")
    bmode = _REDUCTIONS[batch_reduction]
    dev = x.device
    with torch.cuda.device(dev):
        dx = torch.empty((B, P1), dtype=torch.float32, device=dev)
        ix = torch.empty((B, P1), dtype=torch.int64, device=dev)
        dy = iy = None
        if not single_directional:
            dy = torch.empty((B, P2), dtype=torch.float32, device=dev)
            iy = torch.empty((B, P2), dtype=torch.int64, device=dev)
        loss = torch.empty((B,) if bmode == PC_REDUCTION_NONE else (), dtype=torch.float32,
                           device=dev)
        st = lib().pc_chamfer(
            x.data_ptr() if P1 > 0 else None, B, P1,
            y.data_ptr() if P2 > 0 else None, P2, _ptr_or_none(xl),
            _ptr_or_none(yl), _ptr_or_none(weights),
            _REDUCTIONS[point_reduction], bmode, int(bool(single_directional)),
            dx.data_ptr() if dx.numel() else None,
            ix.data_ptr() if ix.numel() else None,
            dy.data_ptr() if dy is not None and dy.numel() else None,
            iy.data_ptr() if iy is not None and iy.numel() else None,
            loss.data_ptr() if loss.numel() else None, _stream_ptr(dev))
    _raise_on(st, "pc_chamfer")
    return loss, (dx, ix), (None if single_directional else (dy, iy))


def pc_three_interpolate(features: torch.Tensor, idx: torch.Tensor,
                         weight: torch.Tensor, *, out: torch.Tensor | None = None):
    """out[b,c,i] = sum_t weight[b,i,t] * features[b,c,idx[b,i,t]] -> [B,C,n]."""
    _check_interp(features, idx, weight)
    B, C, M = features.shape
    n = idx.shape[1]
    with torch.cuda.device(features.device):
        if out is None:
            out = torch.empty((B, C, n), dtype=torch.float32, device=features.device)
        st = lib().pc_three_interpolate(features.data_ptr() if M > 0 else None,
                                        B, C, M, idx.data_ptr(), weight.data_ptr(),
                                        n, out.data_ptr(),
                                        _stream_ptr(features.device))
    _raise_on(st, "pc_three_interpolate")
    return out


def pc_three_interpolate_backward(grad_out: torch.Tensor, idx: torch.Tensor,
                                  weight: torch.Tensor, M: int, *,
                                  out: torch.Tensor | None = None):
    """Gradient of three_interpolate w.r.t. the features: [B,C,n] -> [B,C,M]."""
    if grad_out.device.type != "cuda" or grad_out.dtype != torch.float32 \
            or grad_out.dim() != 3 or not grad_out.is_contiguous():
        raise ValueError("grad_out must be a contiguous float32 CUDA tensor [B,C,n]")
    B, C, n = grad_out.shape
    _check_triplets(idx, weight, B, n, grad_out.device)
    with torch.cuda.device(grad_out.device):
        if out is None:
            out = torch.empty((B, C, M), dtype=torch.float32, device=grad_out.device)
        st = lib().pc_three_interpolate_backward(
            grad_out.data_ptr() if grad_out.numel() else None, B, C, n,
            idx.data_ptr() if idx.numel() else None,
            weight.data_ptr() if weight.numel() else None, M,
            out.data_ptr() if out.numel() else None, _stream_ptr(grad_out.device))
    _raise_on(st, "pc_three_interpolate_backward")
    return out


def _check_triplets(idx, weight, B, n, device):
    if idx.device != device or weight.device != device:
        raise ValueError("idx and weight must be on the features' device")
    if idx.dtype != torch.int64 or tuple(idx.shape) != (B, n, 3) or not idx.is_contiguous():
        raise ValueError(f"idx must be a contiguous int64 tensor [{B}, {n}, 3]")
    if weight.dtype != torch.float32 or tuple(weight.shape) != (B, n, 3) \
            or not weight.is_contiguous():
        raise ValueError(f"weight must be a contiguous float32 tensor [{B}, {n}, 3]")


def _check_interp(features, idx, weight):
    if not isinstance(features, torch.Tensor) or features.device.type != "cuda":
        raise ValueError("features must be a CUDA tensor; this library has no CPU path")
    if features.dtype != torch.float32 or features.dim() != 3 \
            or not features.is_contiguous():
        raise ValueError("features must be a contiguous float32 tensor [B, C, M]")
    B = features.shape[0]
    if idx.dim() != 3:
        raise ValueError("idx must be [B, n, 3]")
    _check_triplets(idx, weight, B, idx.shape[1], features.device)


class _ThreeInterpolate(torch.autograd.Function):
    @staticmethod
    def forward(ctx, features, idx, weight):
        ctx.save_for_backward(idx, weight)
        ctx.M = features.shape[2]
        return pc_three_interpolate(features.contiguous(), idx, weight)

    @staticmethod
    def backward(ctx, grad_out):
        idx, weight = ctx.saved_tensors
        return (pc_three_interpolate_backward(grad_out.contiguous(), idx, weight,
                                              ctx.M), None, None)


def three_nn(unknown: torch.Tensor, known: torch.Tensor):
    """The three nearest known points of every unknown point: (dist, idx),
    Euclidean distances, [B, n, 3] each (pc_knn with k = 3)."""
    return pc_knn(unknown, known, 3)


def three_interpolate(features: torch.Tensor, idx: torch.Tensor,
                      weight: torch.Tensor) -> torch.Tensor:
    """Differentiable (w.r.t. features) three_interpolate: [B,C,M] -> [B,C,n]."""
    return _ThreeInterpolate.apply(features, idx, weight)


def chamfer_distance(x: torch.Tensor, y: torch.Tensor, x_lengths=None,
                     y_lengths=None, weights=None, batch_reduction="mean",
                     point_reduction="mean", single_directional=False):
    """Squared-L2 Chamfer loss, forward only: returns (loss, None) -- the
    second element stands for a normals loss, which is not computed."""
    loss, _, _ = pc_chamfer(x, y, x_lengths=x_lengths, y_lengths=y_lengths,
                            weights=weights, point_reduction=point_reduction,
                            batch_reduction=batch_reduction,
                            single_directional=single_directional)
    return loss, None


def pc_gather_points(xyz: torch.Tensor, idx: torch.Tensor, *,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """out[b,q,t,:] = xyz[b, idx[b,q,t], :]; zeros where idx = -1."""
    _check_cloud(xyz, "xyz")
    B, N, _ = xyz.shape
    if idx.device != xyz.device or idx.dtype != torch.int64 or idx.dim() != 3 \
            or idx.shape[0] != B or not idx.is_contiguous():
        raise ValueError("idx must be a contiguous int64 CUDA tensor [B, Q, K]")
    Q, K = idx.shape[1], idx.shape[2]
    with torch.cuda.device(xyz.device):
        if out is None:
            out = torch.empty((B, Q, K, 3), dtype=torch.float32, device=xyz.device)
        st = lib().pc_gather_points(xyz.data_ptr() if N > 0 else None, B, N,
                                    idx.data_ptr() if idx.numel() else None, Q, K,
                                    out.data_ptr() if out.numel() else None,
                                    _stream_ptr(xyz.device))
    _raise_on(st, "pc_gather_points")
    return out


def pc_device_status(reset: bool = True, device=None) -> int:
    """Synchronize the current stream and return (and clear) the status word."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None \
        else torch.device(device)
    out = ctypes.c_int32(0)
    with torch.cuda.device(device):
        st = lib().pc_device_status(_stream_ptr(device), int(reset),
                                    ctypes.byref(out))
    _raise_on(st, "pc_device_status")
    return out.value


def pc_set_wait_timeout_ns(ns: int):
    lib().pc_set_wait_timeout_ns(int(ns))


def pc_debug_set_fps_grid_stall(enable: bool):
    lib().pc_debug_set_fps_grid_stall(int(bool(enable)))


PC_STALL_FPS_GRID, PC_STALL_FPS_CLUSTER, PC_STALL_TILE_STREAM = 1, 2, 4


def pc_debug_set_stall(mask: int):
    """Testing hooks that make a bounded device wait run out (PC_STALL_*
    flags; 0 restores normal operation)."""
    lib().pc_debug_set_stall(int(mask))


def pc_fps_set_batched(enable: bool) -> bool:
    """FPS in rounds of several centers per exchange (default) or one center
    per exchange; returns the previous setting.  Results do not depend on
    it."""
    return bool(lib().pc_fps_set_batched(1 if enable else 0))


def pc_set_sm_reserve(sms: int):
    """SMs that concurrent work on another stream occupies (a planning hint
    for the brute-force kNN grid; results do not depend on it)."""
    lib().pc_set_sm_reserve(int(sms))


def pc_fps_sm_count(B: int, N: int, npoint: int) -> int:
    """SMs an FPS launch of these sizes occupies on the current device."""
    return int(lib().pc_fps_sm_count(int(B), int(N), int(npoint)))


def pc_fps_plan(B: int, N: int, strategy: int = PC_FPS_AUTO, cluster_size: int = 0,
                blocks_per_cloud: int = 0):
    """(strategy, cluster size, blocks per cloud) of the FPS schedule for
    these sizes on the current device."""
    st, cs, bpc = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    _raise_on(lib().pc_fps_plan(int(B), int(N), int(strategy), int(cluster_size),
                                int(blocks_per_cloud), ctypes.byref(st),
                                ctypes.byref(cs), ctypes.byref(bpc)), "pc_fps_plan")
    return st.value, cs.value, bpc.value


# mps-pointops-style names
def furthest_point_sample(xyz, npoint, start_idx=0):
    return pc_fps(xyz, npoint, start_idx)


def knn(query, ref, k):
    return pc_knn(query, ref, k)


def ball_query(query, ref, radius, K):
    return pc_ball_query(query, ref, radius, K)
