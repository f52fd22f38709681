"""PyTorch3D-style Ball Query adapter over the dense first-K Ball Query.

mps-pointops project page, "PyTorch3D-style Ball Query": the PyTorch3D
argument order and defaults (p1, p2, lengths1, lengths2, K=500, radius=0.2,
return_nn=True, skip_points_outside_cube), returning KNN(dists, idx, knn)
with zero coordinates in knn where idx = -1 and knn = None when return_nn is
False.  The cube flag is a result-preserving hint and does not change the
search.  Only three-dimensional float32 coordinates are supported.

Argument marshalling only: the search is pc_ball_query_ex and the neighbor
coordinates come from pc_gather_points (both CUDA kernels of
libpointcloud.so).  It is an explicit adapter; it does not register itself
as, or replace, a PyTorch3D installation.
"""
from __future__ import annotations

from collections import namedtuple

import torch

from .binding import pc_ball_query, pc_gather_points

KNN = namedtuple("KNN", ["dists", "idx", "knn"])


def ball_query(p1: torch.Tensor, p2: torch.Tensor,
               lengths1: torch.Tensor | None = None,
               lengths2: torch.Tensor | None = None, K: int = 500,
               radius: float = 0.2, return_nn: bool = True,
               skip_points_outside_cube: bool = False) -> KNN:
    """For every point of p1 [N, P1, 3], the first K points of p2 [N, P2, 3]
    (in index order) with squared distance < fl32(radius)^2.

    Returns KNN(dists [N,P1,K] squared distances, idx [N,P1,K] int64 with -1
    padding, knn [N,P1,K,3] neighbor coordinates or None).  lengths1 /
    lengths2 ([N] int64) mask padded points of each cloud.
    """
    del skip_points_outside_cube  # hint only: the results do not depend on it
    if lengths1 is not None:
        lengths1 = lengths1.to(device=p1.device, dtype=torch.int64).contiguous()
    if lengths2 is not None:
        lengths2 = lengths2.to(device=p1.device, dtype=torch.int64).contiguous()
    dists, idx = pc_ball_query(p1, p2, float(radius), int(K),
                               query_lengths=lengths1, ref_lengths=lengths2)
    nn = pc_gather_points(p2, idx) if return_nn else None
    return KNN(dists=dists, idx=idx, knn=nn)
