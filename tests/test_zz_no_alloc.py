"""pc_fps_grid_static: FPS for callers that cannot allocate device memory.

Such callers (a program whose device memory all belongs to its own pool, or
a fixed-footprint real-time loop) cannot let the library allocate scratch,
nor allocate a workspace for it.  This entry point keeps the grid schedule's
scratch in a fixed array inside the library.  The test calls it through the
C ABI twice in a row -- on two different clouds, so the second call runs on
whatever the first left in the array -- and compares each result with the
regular entry point (pc_fps_ex, grid schedule, library-allocated scratch) and
with the oracle.  Indices must be identical.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
from point_cloud_neighbor_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _regular(x, npoint, start, bpc):
    return binding.pc_fps(x, npoint, start, strategy=binding.PC_FPS_GRID,
                          blocks_per_cloud=bpc)


def _static(x, npoint, start, bpc):
    L = binding.lib()
    B, N, _ = x.shape
    out = torch.full((B, npoint), -7, dtype=torch.int64, device=x.device)
    st = L.pc_fps_grid_static(x.data_ptr(), B, N, npoint, start, out.data_ptr(),
                              bpc, torch.cuda.current_stream(x.device).cuda_stream)
    assert st == 0, L.pc_last_error_message().decode()
    return out


def test_static_scratch_fps_matches_regular_entry_point_twice():
    dev = torch.device("cuda:0")
    first = inputs.large()                                  # 1 x 100k
    second = inputs.random_cloud(21, 2, 7001)
    for xh, npoint, start, bpc in ((first, 1000, 5, 0), (second, 600, 3, 9)):
        x = torch.from_numpy(xh).to(dev)
        want = _regular(x, npoint, start, bpc)
        got = _static(x, npoint, start, bpc)
        torch.cuda.synchronize(dev)
        g, w = got.cpu().numpy(), want.cpu().numpy()
        assert np.array_equal(g, w), f"{int((g != w).sum())} of {g.size} indices differ"
        o = oracle.fps(xh, npoint, start, threads=oracle.default_threads())
        assert np.array_equal(g, o), f"{int((g != o).sum())} of {g.size} differ from the oracle"
    assert binding.pc_device_status(reset=True) == 0


def test_static_scratch_rejects_bad_arguments():
    L = binding.lib()
    x = torch.from_numpy(inputs.random_cloud(22, 1, 100)).to("cuda:0")
    out = torch.empty((1, 4), dtype=torch.int64, device="cuda:0")
    assert L.pc_fps_grid_static(x.data_ptr(), 1, 100, 4, 100, out.data_ptr(), 0,
                                None) == binding.PC_ERR_INVALID_ARGUMENT
    assert L.pc_fps_grid_static(x.data_ptr(), 1, 100, 0, 0, out.data_ptr(), 0,
                                None) == binding.PC_ERR_INVALID_ARGUMENT
