"""Host-side checks of the C ABI that need no GPU.

The library must load, export every function include/pointcloud.h declares,
and reject invalid arguments on the host (before touching any device) with
the documented status codes.  With no usable device, a valid call reports
PC_ERR_NO_DEVICE -- never a silent CPU result.
"""
import ctypes
import os
import re

import pytest
import torch

from point_cloud_neighbor_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pointcloud.h")


@pytest.fixture(scope="module")
def L():
    from point_cloud_neighbor_gb300 import build
    build.build()
    return binding.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pc_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_three_operators():
    names = header_functions()
    for n in ("pc_fps", "pc_knn", "pc_ball_query"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in header_functions():
        assert hasattr(L, name), f"{name} declared but not exported"
    assert set(header_functions()) == set(binding.exported_symbols())


def test_status_strings(L):
    assert L.pc_status_string(0) == b"PC_OK"
    assert L.pc_status_string(1) == b"PC_ERR_INVALID_ARGUMENT"
    assert L.pc_status_string(2) == b"PC_ERR_UNSUPPORTED"
    assert L.pc_status_string(3) == b"PC_ERR_CUDA"
    assert L.pc_status_string(4) == b"PC_ERR_DEVICE_TIMEOUT"
    assert L.pc_status_string(5) == b"PC_ERR_NO_DEVICE"
    assert L.pc_status_string(99) == b"PC_ERR_UNKNOWN"
    assert L.pc_version() >= 100


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first


def _msg(L):
    return L.pc_last_error_message().decode()


def test_knn_k_above_n_is_invalid(L):
    st = L.pc_knn(FAKE, 1, 4, FAKE, 3, 4, FAKE, FAKE, None)
    assert st == binding.PC_ERR_INVALID_ARGUMENT
    assert "k <= N" in _msg(L)


def test_knn_k_zero_and_negative_sizes_invalid(L):
    assert L.pc_knn(FAKE, 1, 4, FAKE, 8, 0, FAKE, FAKE, None) == 1
    assert L.pc_knn(FAKE, -1, 4, FAKE, 8, 2, FAKE, FAKE, None) == 1
    assert L.pc_knn(FAKE, 1, -4, FAKE, 8, 2, FAKE, FAKE, None) == 1


def test_knn_k_above_compiled_max_unsupported(L):
    st = L.pc_knn(FAKE, 1, 4, FAKE, 1000, 257, FAKE, FAKE, None)
    assert st == binding.PC_ERR_UNSUPPORTED


def test_knn_empty_batch_is_ok_without_device(L):
    assert L.pc_knn(None, 0, 4, None, 8, 2, None, None, None) == 0
    assert L.pc_knn(None, 2, 0, None, 8, 2, None, None, None) == 0


@pytest.mark.parametrize("radius", [0.0, -1.0, float("nan"), float("inf")])
def test_ball_query_bad_radius_invalid(L, radius):
    st = L.pc_ball_query(FAKE, 1, 1, FAKE, 4, radius, 2, FAKE, FAKE, None)
    assert st == binding.PC_ERR_INVALID_ARGUMENT


def test_ball_query_bad_K_invalid(L):
    assert L.pc_ball_query(FAKE, 1, 1, FAKE, 4, 0.5, 0, FAKE, FAKE, None) == 1


def test_fps_bad_arguments(L):
    o = FAKE
    assert L.pc_fps(FAKE, 1, 4, 0, 0, o, None, 0, None) == 1        # npoint 0
    assert L.pc_fps(FAKE, 1, 4, 2, 4, o, None, 0, None) == 1        # start == N
    assert L.pc_fps(FAKE, 1, 4, 2, -1, o, None, 0, None) == 1       # start < 0
    assert L.pc_fps(FAKE, 1, 0, 2, 0, o, None, 0, None) == 1        # N = 0
    assert L.pc_fps_ex(FAKE, 1, 4, 2, 0, o, None, 0, 7, 0, 0, None) == 1
    assert L.pc_fps_ex(FAKE, 1, 4, 2, 0, o, None, 0, 2, 17, 0, None) == 1
    assert L.pc_fps(None, 0, 4, 2, 0, None, None, 0, None) == 0     # B = 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_valid_call_without_device_reports_no_device(L):
    st = L.pc_knn(FAKE, 1, 4, FAKE, 8, 2, FAKE, FAKE, None)
    assert st == binding.PC_ERR_NO_DEVICE
    st = L.pc_ball_query(FAKE, 1, 1, FAKE, 4, 0.5, 2, FAKE, FAKE, None)
    assert st == binding.PC_ERR_NO_DEVICE
    st = L.pc_fps(FAKE, 1, 4, 2, 0, FAKE, None, 0, None)
    assert st == binding.PC_ERR_NO_DEVICE
    assert L.pc_fps_workspace_bytes(1, 1_000_000, 16) == 0


def test_binding_rejects_cpu_tensors(L):
    x = torch.zeros(1, 8, 3)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.pc_fps(x, 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.pc_knn(x, x, 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        binding.pc_ball_query(x, x, 0.5, 2)


def test_wait_timeout_setter_accepts_any_value(L):
    L.pc_set_wait_timeout_ns(0)
    L.pc_set_wait_timeout_ns(2_000_000_000)
    L.pc_debug_set_fps_grid_stall(0)
    for mask in (1, 2, 4, 7, 0):
        L.pc_debug_set_stall(mask)


def test_sm_reserve_and_fps_sm_count_without_device(L):
    # the reserve is a host-side hint: any value is taken (negative as 0)
    L.pc_set_sm_reserve(-5)
    L.pc_set_sm_reserve(16)
    L.pc_set_sm_reserve(0)
    # no device here: the FPS footprint is unknown (0), as for empty sizes
    assert L.pc_fps_sm_count(1, 100000, 4096) == 0
    assert L.pc_fps_sm_count(0, 100000, 4096) == 0
    assert L.pc_fps_sm_count(1, 0, 4096) == 0


def test_fps_plan_without_device(L):
    import ctypes
    st, cs, bpc = ctypes.c_int(7), ctypes.c_int(7), ctypes.c_int(7)
    assert L.pc_fps_plan(1, 100000, 0, 0, 0, None, None, None) == 1
    assert L.pc_fps_plan(0, 100000, 0, 0, 0, ctypes.byref(st), ctypes.byref(cs),
                         ctypes.byref(bpc)) == 1
    assert (st.value, cs.value, bpc.value) == (0, 0, 0)
    # sizes are valid, but there is no device to plan for
    assert L.pc_fps_plan(1, 100000, 0, 0, 0, ctypes.byref(st), ctypes.byref(cs),
                         ctypes.byref(bpc)) == 5


def test_knn_ex_validation(L):
    # k > N is allowed in the ex form (padded); k above 256 is unsupported
    assert L.pc_knn_ex(None, 0, 4, None, 8, 300, None, None, 0, None, None, None) == 2
    assert L.pc_knn_ex(FAKE, 1, 4, FAKE, 8, 0, None, None, 0, FAKE, FAKE, None) == 1
    assert L.pc_knn_ex(FAKE, 1, 4, FAKE, 8, 2, None, None, 4, FAKE, FAKE, None) == 1
    assert "unknown flags" in _msg(L)
    assert L.pc_knn_ex(None, 0, 4, None, 3, 5, None, None, 1, None, None, None) == 0


def test_ball_query_ex_validation(L):
    assert L.pc_ball_query_ex(FAKE, 1, 1, FAKE, 4, None, None, -1.0, 2, FAKE, FAKE,
                              None) == 1
    assert L.pc_ball_query_ex(FAKE, 1, 1, FAKE, 4, None, None, 0.5, 0, FAKE, FAKE,
                              None) == 1
    assert L.pc_ball_query_ex(None, 2, 0, None, 4, None, None, 0.5, 3, None, None,
                              None) == 0


def test_chamfer_validation(L):
    args = (FAKE, 1, 4, FAKE, 4, None, None, None)
    outs = (FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert L.pc_chamfer(FAKE, -1, 4, FAKE, 4, None, None, None, 2, 2, 0, *outs) == 1
    assert L.pc_chamfer(*args, 0, 2, 0, *outs) == 1     # point reduction NONE
    assert "point_reduction" in _msg(L)
    assert L.pc_chamfer(*args, 2, 7, 0, *outs) == 1     # unknown batch reduction
    assert L.pc_chamfer(FAKE, 70000, 4, FAKE, 4, None, None, None, 2, 2, 0,
                        *outs) == 2
    # B = 0 without a reduced loss: nothing to do
    assert L.pc_chamfer(None, 0, 4, None, 4, None, None, None, 2, 0, 0,
                        None, None, None, None, None, None) == 0


def test_interp_and_gather_validation(L):
    assert L.pc_three_interpolate(FAKE, -1, 2, 3, FAKE, FAKE, 4, FAKE, None) == 1
    assert L.pc_three_interpolate(FAKE, 70000, 2, 3, FAKE, FAKE, 4, FAKE, None) == 2
    assert L.pc_three_interpolate(None, 0, 2, 3, None, None, 4, None, None) == 0
    assert L.pc_three_interpolate_backward(FAKE, 1, 2, -4, FAKE, FAKE, 3, FAKE,
                                           None) == 1
    assert L.pc_three_interpolate_backward(None, 2, 0, 4, None, None, 3, None,
                                           None) == 0
    assert L.pc_gather_points(FAKE, 1, -1, FAKE, 2, 2, FAKE, None) == 1
    assert L.pc_gather_points(None, 1, 5, None, 0, 3, None, None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_new_entry_points_report_no_device(L):
    assert L.pc_knn_ex(FAKE, 1, 4, FAKE, 8, 2, None, None, 0, FAKE, FAKE,
                       None) == binding.PC_ERR_NO_DEVICE
    assert L.pc_chamfer(FAKE, 1, 4, FAKE, 4, None, None, None, 2, 2, 0,
                        FAKE, FAKE, FAKE, FAKE, FAKE, None) == binding.PC_ERR_NO_DEVICE
    assert L.pc_three_interpolate(FAKE, 1, 2, 3, FAKE, FAKE, 4, FAKE,
                                  None) == binding.PC_ERR_NO_DEVICE
    assert L.pc_gather_points(FAKE, 1, 5, FAKE, 2, 2, FAKE,
                              None) == binding.PC_ERR_NO_DEVICE


def test_pytorch3d_adapter_rejects_cpu_tensors(L):
    from point_cloud_neighbor_gb300.pytorch3d import ball_query
    x = torch.zeros(1, 8, 3)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ball_query(x, x, K=4, radius=0.5)
