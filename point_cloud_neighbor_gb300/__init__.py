"""GB300-native dense point-cloud neighbor search (FPS, kNN, Ball Query) and
the operators built on it (exact grid search, Chamfer distance, PointNet++
feature propagation, neighbor gather).

The compute lives in libpointcloud.so (CUDA kernels for sm_103a behind the C
ABI of include/pointcloud.h); this package holds its ctypes binding, the
build script, the PyTorch3D-style Ball Query adapter (``.pytorch3d``) and the
seeded workload generators.
"""
from .binding import (PC_FPS_AUTO, PC_FPS_BLOCK, PC_FPS_CLUSTER, PC_FPS_GRID,
                      PointCloudError, PointGrid, ball_query, chamfer_distance,
                      furthest_point_sample, knn, pc_ball_query,
                      pc_ball_query_grid, pc_chamfer,
                      pc_debug_set_fps_grid_stall, pc_debug_set_stall,
                      PC_STALL_FPS_GRID, PC_STALL_FPS_CLUSTER, PC_STALL_TILE_STREAM,
                      pc_device_status, pc_fps,
                      pc_gather_points, pc_grid_build, pc_knn, pc_knn_d,
                      pc_knn_ball_query, pc_knn_ball_query_plan,
                      pc_fps_set_batched,
                      pc_knn_grid,
                      pc_set_wait_timeout_ns, pc_set_sm_reserve,
                      pc_fps_sm_count, pc_fps_plan, pc_three_interpolate,
                      pc_three_interpolate_backward, three_interpolate,
                      three_nn)

__all__ = [
    "PC_FPS_AUTO", "PC_FPS_BLOCK", "PC_FPS_CLUSTER", "PC_FPS_GRID",
    "PointCloudError", "ball_query", "furthest_point_sample", "knn",
    "pc_ball_query", "pc_debug_set_fps_grid_stall", "pc_device_status",
    "pc_fps", "pc_knn", "pc_set_wait_timeout_ns", "PointGrid",
    "pc_grid_build", "pc_knn_grid", "pc_ball_query_grid", "pc_chamfer",
    "chamfer_distance", "pc_three_interpolate", "pc_three_interpolate_backward",
    "three_interpolate", "three_nn", "pc_gather_points", "pc_knn_d",
    "pc_set_sm_reserve", "pc_fps_sm_count", "pc_fps_plan", "pc_debug_set_stall",
    "PC_STALL_FPS_GRID", "PC_STALL_FPS_CLUSTER", "PC_STALL_TILE_STREAM",
    "pc_knn_ball_query", "pc_knn_ball_query_plan", "pc_fps_set_batched",
]
