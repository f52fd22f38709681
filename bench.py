"""Benchmark: one step = FPS + kNN + Ball Query on the 100k-point workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Workload (the single-large-cloud configuration): B=1, N=100,000 points from a
mixture of 64 isotropic Gaussians (sigma 0.05, means uniform in [0,1)^3),
random order.  One step runs, on inputs already resident in device memory:
  * farthest point sampling of 4,096 centers from index 0,
  * kNN with k=16 of all 100,000 points against all 100,000,
  * Ball Query r=0.02, K=32 of all 100,000 points against all 100,000.
Headline ``value``: (kNN queries + Ball Query queries) per second of whole
steps (FPS time included in the step time); per-operator throughputs
(queries/s, samples/s) and roofline fractions are in ``ops``.

Timing: W untimed warm-up steps, then K steps, each preceded by an L2 flush
(a 512 MiB device write outside the timed events) and bracketed by CUDA
events on the launching stream; a barrier + synchronize brackets the whole
timed loop; the max over ranks is reported.  With N > 1 (torchrun) every rank
runs its own replica of the workload on its own GPU (the three operators
have no cross-GPU exchange step): value = N * units / max time, scaling
"weak".

``--impl reference`` times the CPU oracle (the plain restatement of the
operator definitions that the parity tests use) on the host cores, on a
bounded sample of the same workload per step, and reports the same metric
extrapolated to the full step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "kNN & Ball Query queries/s, FPS samples/s at 100k pts; % of FP32/HBM roofline"
UNIT = "queries/s"
WORKLOAD = dict(name="large", B=1, N=100_000, npoint=4096, start_idx=0,
                knn_k=16, bq_radius=0.02, bq_K=32, order="random")
FLOPS_PER_PAIR = 8          # 3 sub + 3 mul + 2 add per (query, reference) pair
FPS_BYTES_PER_POINT_STEP = 20  # 12 B coordinates + 4 B min read + 4 B write
L2_FLUSH_BYTES = 512 << 20
# Thread-block cluster FPS runs on in the step.  FPS alone plans 16 blocks;
# next to kNN and Ball Query a 13-block cluster balances the step better:
# FPS still ends first, and the three SMs it gives back go to the Ball Query
# grid (GB300: step 4.27 ms with 13 or 12 blocks, 4.31 with 14, 4.34 with 16;
# FPS alone 3.34 ms with 13 blocks, 3.72 with 16, same samples).
STEP_FPS_CLUSTER = 13


def workload_config(extra=None):
    cfg = {
        "workload": ("single large cloud: B=1, N=100000 fp32 points, mixture of "
                     "64 Gaussians (sigma 0.05), random order; FPS npoint=4096 "
                     "start 0; kNN k=16, 100000 queries vs 100000; Ball Query "
                     "r=0.02 K=32, 100000 queries vs 100000"),
        "B": 1, "N": 100000, "fps_npoint": 4096, "knn_k": 16, "knn_queries": 100000,
        "bq_radius": 0.02, "bq_K": 32, "bq_queries": 100000, "seed": 3,
        "l2": "flushed between timed steps (512 MiB device write outside the events)",
    }
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# distributed helpers (torchrun: one rank per GPU)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(values, world, device=None):
    """Element-wise max of a list of floats over all ranks."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# GPU clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            f = [v.strip() for v in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}, "fallback"


def fp32_alu_peak_tflops(sm_count: int, mhz: float) -> float:
    """FP32 CUDA-core peak counting an FMA as 2 flops: SMs x 128 lanes x 2 x clock."""
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


# The sources each operator's kernel is compiled from (its .cu file and the
# headers it includes); a recorded DRAM figure is used only while they are
# unchanged.
KERNEL_SOURCES = {
    "knn": ["pc_knn.cu", "pc_device.cuh", "pc_filter.cuh", "pc_stream.cuh",
            "pc_tiles.cuh"],
    "ball_query": ["pc_ball_query.cu", "pc_device.cuh", "pc_filter.cuh",
                   "pc_stream.cuh", "pc_tiles.cuh"],
    "fps": ["pc_fps.cu", "pc_device.cuh"],
    "knn_ball_query": ["pc_knn.cu", "pc_device.cuh", "pc_filter.cuh", "pc_stream.cuh",
                       "pc_tiles.cuh"],
    "grid_knn": ["pc_grid.cu", "pc_device.cuh"],
    "grid_ball_query": ["pc_grid.cu", "pc_device.cuh"],
}


def kernel_source_hash(op: str) -> str:
    """Hash of the code of an operator's sources: line comments, trailing
    blanks and blank lines do not count, so that editing a comment keeps a
    capture valid while any change of code does not."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[op]:
        with open(os.path.join(ROOT, "point_cloud_neighbor_gb300", "csrc", name),
                  encoding="utf-8") as fh:
            for line in fh:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(op: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(op)
    for line in open(path):
        if line.startswith("#"):  # the header: the capture command
            continue
        kv = dict(p.split("=", 1) for p in line.split() if "=" in p)
        if kv.get("op") == op and kv.get("src_sha256") == want:
            try:
                return float(kv["dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        init_dist(world, "nccl")
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)

    import point_cloud_neighbor_gb300 as pc
    from point_cloud_neighbor_gb300 import inputs

    W = WORKLOAD
    x_host = inputs.large(seed=3, morton=False)        # [1, N, 3] float32
    x = torch.from_numpy(x_host).to(device)
    B, N = 1, W["N"]
    npoint, k, r, K = W["npoint"], W["knn_k"], W["bq_radius"], W["bq_K"]
    stream = torch.cuda.current_stream(device)

    fps_out = torch.empty((B, npoint), dtype=torch.int64, device=device)
    knn_d = torch.empty((B, N, k), dtype=torch.float32, device=device)
    knn_i = torch.empty((B, N, k), dtype=torch.int64, device=device)
    bq_d = torch.empty((B, N, K), dtype=torch.float32, device=device)
    bq_i = torch.empty((B, N, K), dtype=torch.int64, device=device)
    ws_bytes = pc.binding.lib().pc_fps_workspace_bytes(B, N, npoint)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    # FPS runs one thread-block cluster per cloud (STEP_FPS_CLUSTER SMs) for
    # thousands of dependent steps; kNN and Ball Query are independent of it and fill
    # the other SMs.  FPS is issued first, on the main stream, so that its
    # cluster is resident before the kNN and Ball Query blocks (issued on a
    # side stream after the same start point) occupy the rest of the GPU
    # (--serial: everything on one stream).
    side = torch.cuda.Stream(device) if not args.serial else stream
    fork = torch.cuda.Event()
    # the kNN and Ball Query grids (one wave) are planned around the SMs
    # FPS holds while it runs
    reserve = 0 if args.serial else B * args.fps_cluster
    # kNN and Ball Query of the same queries: one fused call (each pair
    # filtered once for both), or with --separate pc_knn then pc_ball_query
    fused = not args.separate

    def step(ev=None):
        # ev: [start, fps_end, knn_start (side), knn_end, bq_end, step_end]
        # (fused: knn_end = bq_end, the end of the one call)
        if ev is not None:
            ev[0].record(stream)
        fork.record(stream)
        pc.pc_fps(x, npoint, 0, strategy=pc.PC_FPS_CLUSTER, cluster_size=args.fps_cluster,
                  out=fps_out, workspace=ws)
        if ev is not None:
            ev[1].record(stream)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            if ev is not None:
                ev[2].record(side)
            pc.pc_set_sm_reserve(reserve)
            if fused:
                pc.pc_knn_ball_query(x, x, k, r, K, out=(knn_d, knn_i, bq_d, bq_i))
            else:
                pc.pc_knn(x, x, k, out_dist=knn_d, out_idx=knn_i)
            if ev is not None:
                ev[3].record(side)
            if not fused:
                pc.pc_ball_query(x, x, r, K, out_dist2=bq_d, out_idx=bq_i)
            pc.pc_set_sm_reserve(0)
            if ev is not None:
                ev[4].record(side)
        stream.wait_stream(side)
        if ev is not None:
            ev[5].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    assert pc.pc_device_status(reset=True, device=device) == 0

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(6)]
              for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    with ClockSampler(device.index if world == 1 else local) as clocks:
        for s in range(args.steps):
            flush.zero_()
            step(events[s])
        torch.cuda.synchronize(device)
    wall1 = time.perf_counter()
    barrier(world)
    # kernels of one step: FPS 1; kNN on this cloud (spatially ordered: the
    # query set is the reference set) frame, count, chunk sums, scan,
    # scatter, seed and the lane kernel = 7 (plus a memset of the cell
    # counts); Ball Query 1 (fused: the kernel that sorts its hits into rows)
    launches = (1 + 7 + 1) * args.steps

    # each operator timed on the stream it runs on
    t_fps = [e[0].elapsed_time(e[1]) for e in events]
    t_knn = [e[2].elapsed_time(e[3]) for e in events]
    t_bq = [e[3].elapsed_time(e[4]) for e in events]
    total_ms = sum(e[0].elapsed_time(e[5]) for e in events)
    total_ms, fps_ms, knn_ms, bq_ms = max_over_ranks(
        [total_ms, sum(t_fps), sum(t_knn), sum(t_bq)], world, device)
    ms_per_step = total_ms / args.steps
    units = (N + N) * world               # kNN + Ball Query queries, all ranks
    value = units / (ms_per_step / 1e3)

    # algorithmic work of each launch
    bq_idx = bq_i.cpu().numpy().reshape(N, K)
    last = bq_idx[:, K - 1]
    bq_pairs = float(np.where(last >= 0, last + 1, N).sum())   # first-K scan length
    # the same scan rounded up to whole blocks of 32 references
    bq_pairs_32 = float(np.minimum(N, 32 * ((np.where(last >= 0, last + 1, N) + 31) // 32)).sum())
    knn_pairs = float(N) * float(N)
    fps_bytes = float(N) * (npoint - 1) * FPS_BYTES_PER_POINT_STEP

    peaks, peak_kind = measured_peaks()
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    clk = clocks.summary()
    max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    alu_peak = fp32_alu_peak_tflops(sm_count, max_mhz)

    if fused:
        per = {"fps": fps_ms / args.steps, "knn_ball_query": (knn_ms + bq_ms) / args.steps}
        # each operator alone, outside the timed step, on the SMs FPS leaves
        # (context: the separate kernels' fractions)
        pc.pc_set_sm_reserve(reserve)
        try:
            per["knn"] = _timed(lambda: pc.pc_knn(x, x, k, out_dist=knn_d, out_idx=knn_i),
                                5, 3, flush, stream)
            per["ball_query"] = _timed(
                lambda: pc.pc_ball_query(x, x, r, K, out_dist2=bq_d, out_idx=bq_i),
                5, 3, flush, stream)
        finally:
            pc.pc_set_sm_reserve(0)
        # and on every SM (each kernel's own fraction of the GPU)
        per["knn_all_sms"] = _timed(
            lambda: pc.pc_knn(x, x, k, out_dist=knn_d, out_idx=knn_i), 5, 3, flush, stream)
        per["ball_query_all_sms"] = _timed(
            lambda: pc.pc_ball_query(x, x, r, K, out_dist2=bq_d, out_idx=bq_i),
            5, 3, flush, stream)
    else:
        per = {"fps": fps_ms / args.steps, "knn": knn_ms / args.steps,
               "ball_query": bq_ms / args.steps}
    ops = {
        "fps": {
            "samples_per_s": npoint * world / (per["fps"] / 1e3),
            "ms": per["fps"],
            "us_per_sample": per["fps"] * 1e3 / (npoint - 1),
            # what a kernel streaming coordinates and minima through HBM every
            # step would move; this one keeps them on chip (context only)
            "streamed_equivalent_gbs": fps_bytes / (per["fps"] / 1e3) / 1e9,
        },
        "knn": {
            "queries_per_s": N * world / (per["knn"] / 1e3),
            "ms": per["knn"], "pairs": knn_pairs,
            "achieved_tflops": knn_pairs * FLOPS_PER_PAIR / (per["knn"] / 1e3) / 1e12,
        },
        "ball_query": {
            "queries_per_s": N * world / (per["ball_query"] / 1e3),
            "ms": per["ball_query"], "pairs": bq_pairs, "pairs_blocks_of_32": bq_pairs_32,
            "achieved_tflops": bq_pairs * FLOPS_PER_PAIR / (per["ball_query"] / 1e3) / 1e12,
        },
    }
    if fused:
        for op, pairs in (("knn", knn_pairs), ("ball_query", bq_pairs)):
            ops[op]["timed"] = "alone on the SMs FPS leaves, outside the timed step"
            ops[op]["sms_used"] = sm_count - reserve
            ops[op]["ms_all_sms"] = per[op + "_all_sms"]
            ops[op]["achieved_tflops_all_sms"] = (
                pairs * FLOPS_PER_PAIR / (per[op + "_all_sms"] / 1e3) / 1e12)
        t_fused = per["knn_ball_query"] / 1e3
        ops["knn_ball_query"] = {
            "queries_per_s": 2 * N * world / t_fused,
            "ms": per["knn_ball_query"], "pairs": knn_pairs + bq_pairs,
            # the two operators' algorithmic work (kNN: every pair; Ball
            # Query: its first-K scan), as for the separate kernels
            "achieved_tflops": (knn_pairs + bq_pairs) * FLOPS_PER_PAIR / t_fused / 1e12,
            # every pair counted once: the work of the one filter pass
            "achieved_tflops_pairs_once": knn_pairs * FLOPS_PER_PAIR / t_fused / 1e12,
            "note": "one pass filters every (query, reference) pair once for both "
                    "operators; achieved_tflops counts both operators' algorithmic "
                    "work (kNN N^2 pairs + the Ball Query first-K scan), "
                    "achieved_tflops_pairs_once the N^2 pairs once",
        }
    # FPS against its two other bounds: ~10 instructions per point-step on the
    # SMs its schedule uses, and the per-step exchange floor measured with the
    # same cluster schedule on 1024 points per block
    fps_sms = B * args.fps_cluster
    ops["fps"]["cluster"] = args.fps_cluster
    ops["fps"]["alu_bound_ms"] = (float(N) * (npoint - 1) * FPS_INSTR_PER_POINT_STEP /
                                  (max(fps_sms, 1) * 128 * max_mhz * 1e6) * 1e3)
    ops["fps"]["alu_frac"] = ops["fps"]["alu_bound_ms"] / per["fps"]
    if fps_sms > 1:
        fx = torch.from_numpy(inputs.random_cloud(7, 1, 1024 * fps_sms)).to(device)
        try:
            floor_ms = _timed(lambda: pc.pc_fps(fx, npoint, 0, strategy=pc.PC_FPS_CLUSTER,
                                                cluster_size=fps_sms),
                              3, 3, flush, stream)
            ops["fps"]["sync_floor_ms"] = floor_ms
            ops["fps"]["sync_floor_frac"] = floor_ms / per["fps"]
            ops["fps"]["sync_floor_note"] = (
                f"the same cluster of {fps_sms} on 1024 points per block, npoint={npoint}")
        except pc.PointCloudError as err:
            ops["fps"]["sync_floor_ms"] = None
            ops["fps"]["sync_floor_note"] = f"not measured: {err}"
    if fused:
        ops["knn_ball_query"]["alu_frac_pairs_once"] = (
            ops["knn_ball_query"]["achieved_tflops_pairs_once"] / alu_peak)
    for op in ("knn", "ball_query") + (("knn_ball_query",) if fused else ()):
        ops[op]["alu_frac_max_clock"] = ops[op]["achieved_tflops"] / alu_peak
        if clk["sm_mhz"]:
            ops[op]["alu_frac_load_clock"] = (
                ops[op]["achieved_tflops"] / fp32_alu_peak_tflops(sm_count, clk["sm_mhz"]))

    def roof_of(op):
        if op == "fps":
            f = ops["fps"]
            floor = f.get("sync_floor_ms")
            r = {"bound": "latency", "achieved": f["us_per_sample"],
                 "peak": floor * 1e3 / (npoint - 1) if floor else None,
                 "unit": "us per step", "frac": (floor / per["fps"]) if floor else None,
                 "alu_frac": f["alu_frac"],
                 "note": "measured floor of the cluster's per-step reduction and "
                         "exchange; points and minima stay on chip (no HBM stream)"}
            r["traffic"] = recorded_traffic(op)
            r["kernel"] = op
            return r
        else:
            r = {"bound": "alu", "achieved": ops[op]["achieved_tflops"],
                 "peak": alu_peak, "unit": "TFLOP/s",
                 "frac": ops[op]["achieved_tflops"] / alu_peak}
            if "alu_frac_pairs_once" in ops[op]:
                r["frac_pairs_once"] = ops[op]["alu_frac_pairs_once"]
            if "sms_used" in ops[op]:
                # against the peak of the SMs it ran on, and alone on all SMs
                r["frac_of_sms_used"] = (ops[op]["achieved_tflops"] /
                                         (alu_peak * ops[op]["sms_used"] / sm_count))
                r["frac_all_sms"] = ops[op]["achieved_tflops_all_sms"] / alu_peak
        r["traffic"] = recorded_traffic(op)
        r["kernel"] = op
        r["peak_source"] = (f"FP32 CUDA cores: {sm_count} SMs x 128 x 2 flop x "
                            f"{max_mhz:.0f} MHz ({peak_kind} max SM clock)"
                            if r["bound"] == "alu" else
                            f"hbm_gbs of MEASURED_PEAKS.json ({peak_kind})")
        return r

    # The dominant kernel is the largest one on the step's critical path: with
    # FPS overlapped, the longer of FPS and the kNN + Ball Query stream;
    # serially, the largest of all.
    side_ops = ("knn_ball_query",) if fused else ("knn", "ball_query")
    side_ms = sum(per[op] for op in side_ops)
    if args.serial:
        candidates, why = ("fps",) + side_ops, "largest kernel of the serial step"
    elif per["fps"] <= side_ms:
        candidates, why = side_ops, ("largest kernel on the step's critical path; "
                                     "FPS runs concurrently with kNN + Ball Query")
    else:
        candidates, why = ("fps",), ("FPS, concurrent with kNN + Ball Query on the "
                                     "other SMs, ends last: the step's critical path")
    dominant = max(candidates, key=per.get)
    roof = roof_of(dominant)
    roof["note"] = why
    roof_all = {op: roof_of(op) for op in ("fps", "knn", "ball_query") + side_ops
                if op in per}

    grid = next_rows = configs = None
    if not args.step_only:
        with_oracle = rank == 0 and world == 1 and not args.no_cpu_baseline
        grid = run_grid(args, pc, x, flush, device, world)
        next_rows = run_next_rows(args, pc, flush, device, world, with_oracle=with_oracle)
        configs = run_configs(args, pc, flush, device, world, with_oracle=with_oracle)

    # end to end through the public API: pinned host in, pinned host out
    e2e = None if args.step_only else run_e2e(args, pc, x_host, device, world)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": workload_config({"parallelism": f"replicas x{world}",
                                   "streams": ("1 (serial)" if args.serial else
                                               "2: FPS concurrent with kNN and Ball Query"),
                                   "knn_ball_query": ("one fused call" if fused else
                                                      "pc_knn then pc_ball_query"),
                                   "fps_cluster": args.fps_cluster}),
        "roofline": roof, "roofline_per_kernel": roof_all, "ops": ops,
        "grid": grid, "next_rows": next_rows, "configs": configs,
        "e2e": e2e,
        "gpu_launches": launches,
        "gpu_launches_note": "the timed FPS + kNN + Ball Query step; the grid and "
                             "next_rows sections are timed separately",
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                   "reasons": clk["reasons"], "samples": clk["samples"]},
        "wall_s_timed_loop": wall1 - wall0,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(x_host, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_only(args):
    """One operator of the step on the workload, W untimed + K timed calls."""
    import torch
    import point_cloud_neighbor_gb300 as pc
    from point_cloud_neighbor_gb300 import inputs
    W = WORKLOAD
    device = torch.device("cuda", 0)
    x = torch.from_numpy(inputs.large(seed=3, morton=False)).to(device)
    g = pc.pc_grid_build(x) if args.only.startswith("grid") else None
    calls = {
        "fps": lambda: pc.pc_fps(x, W["npoint"], 0),
        "knn": lambda: pc.pc_knn(x, x, W["knn_k"]),
        "ball_query": lambda: pc.pc_ball_query(x, x, W["bq_radius"], W["bq_K"]),
        "knn_ball_query": lambda: pc.pc_knn_ball_query(x, x, W["knn_k"], W["bq_radius"],
                                                       W["bq_K"]),
        "grid_build": lambda: pc.pc_grid_build(x),
        "grid_knn": lambda: pc.pc_knn_grid(x, g, W["knn_k"]),
        "grid_ball_query": lambda: pc.pc_ball_query_grid(x, g, W["bq_radius"],
                                                         W["bq_K"]),
    }
    if args.only == "knn_d":
        fx = torch.randn((32, 1024, 64), device=device)
        calls["knn_d"] = lambda: pc.pc_knn_d(fx, fx, 20)
    if args.only in ("fps_1m", "knn_1m", "ball_query_1m"):
        # the 1M-point cloud; queries: 16,384 points spread over it
        vx = torch.from_numpy(inputs.very_large()).to(device)
        vq = vx[:, ::61][:, :16384].contiguous()
        calls["fps_1m"] = lambda: pc.pc_fps(vx, 16384, 0)
        calls["knn_1m"] = lambda: pc.pc_knn(vq, vx, 32)
        calls["ball_query_1m"] = lambda: pc.pc_ball_query(vq, vx, 0.01, 64)
    if args.only in ("chamfer", "three_interpolate", "three_interpolate_backward"):
        cx = torch.from_numpy(inputs.random_cloud(5, 4, 16384)).to(device)
        cy = torch.from_numpy(inputs.random_cloud(6, 4, 16384)).to(device)
        px = torch.from_numpy(inputs.pointnet2()).to(device)
        centers = px[:, :1024].contiguous()
        d, idx = pc.three_nn(px, centers)
        w = (1.0 / (d + 1e-8))
        w = (w / w.sum(-1, keepdim=True)).contiguous()
        feats = torch.randn((16, 256, 1024), device=device)
        gup = torch.randn((16, 256, 4096), device=device)
        calls["chamfer"] = lambda: pc.pc_chamfer(cx, cy)
        calls["three_interpolate"] = lambda: pc.pc_three_interpolate(feats, idx, w)
        calls["three_interpolate_backward"] = lambda: pc.pc_three_interpolate_backward(
            gup, idx, w, 1024)
    fn = calls[args.only]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    ms = _timed(fn, args.steps, args.warmup, flush, torch.cuda.current_stream(device))
    print(json.dumps({"op": args.only, "ms": ms, "calls": args.steps,
                      "l2": "flushed before every call (outside the events)"}))


def run_grid(args, pc, x, flush, device, world):
    """The same kNN and Ball Query through the exact grid path (grid built
    every step, inside the timed events): results equal the brute-force
    kernels'; reported next to them, not as the headline."""
    import torch
    W = WORKLOAD
    N, k, r, K = W["N"], W["knn_k"], W["bq_radius"], W["bq_K"]
    stream = torch.cuda.current_stream(device)
    kd = torch.empty((1, N, k), dtype=torch.float32, device=device)
    ki = torch.empty((1, N, k), dtype=torch.int64, device=device)
    bd = torch.empty((1, N, K), dtype=torch.float32, device=device)
    bi = torch.empty((1, N, K), dtype=torch.int64, device=device)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        g = pc.pc_grid_build(x)
        if ev is not None:
            ev[1].record(stream)
        pc.pc_knn_grid(x, g, k, out_dist=kd, out_idx=ki)
        if ev is not None:
            ev[2].record(stream)
        pc.pc_ball_query_grid(x, g, r, K, out_dist2=bd, out_idx=bi)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    steps = max(3, args.steps)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
              for _ in range(steps)]
    torch.cuda.synchronize(device)
    for s in range(steps):
        flush.zero_()
        step(events[s])
    torch.cuda.synchronize(device)
    b_ms, k_ms, q_ms = max_over_ranks(
        [sum(e[0].elapsed_time(e[1]) for e in events) / steps,
         sum(e[1].elapsed_time(e[2]) for e in events) / steps,
         sum(e[2].elapsed_time(e[3]) for e in events) / steps], world, device)
    return {"build_ms": b_ms, "knn_ms": k_ms, "ball_query_ms": q_ms,
            "knn_queries_per_s": N * world / ((b_ms + k_ms) / 1e3),
            "ball_query_queries_per_s": N * world / ((b_ms + q_ms) / 1e3),
            "queries_per_s": 2 * N * world / ((b_ms + k_ms + q_ms) / 1e3),
            "launches_per_step": 9,
            "note": "exact uniform-grid path (pc_grid_build + pc_knn_grid + "
                    "pc_ball_query_grid), grid rebuilt every step; identical "
                    "results to the brute-force kernels"}


def _timed(fn, steps, warmup, flush, stream):
    """Mean CUDA-event time (ms) of fn() over `steps` calls, L2 flushed
    before each call."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def run_next_rows(args, pc, flush, device, world, with_oracle):
    """The operators built on the hot path, each on the workload the pages
    time it on: Chamfer forward (batch 4, 16,384 points per cloud), the
    PointNet++ feature-propagation three_interpolate (16 clouds, 1024 centers
    -> 4096 points, 256 channels) and the PyTorch3D-style Ball Query (16
    clouds, 1024 centers vs 4096 points, r = 0.2, K = 64, return_nn)."""
    import torch
    from point_cloud_neighbor_gb300 import inputs
    from point_cloud_neighbor_gb300.pytorch3d import ball_query as p3d_ball_query
    stream = torch.cuda.current_stream(device)
    steps, warm = max(3, args.steps), max(3, args.warmup)
    peaks, _ = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    alu = fp32_alu_peak_tflops(sm_count, float(peaks.get("sm_max_mhz", 2070.0)))
    out = {}

    # Chamfer forward
    CB, CP = 4, 16384
    cx_h = inputs.random_cloud(5, CB, CP)
    cy_h = inputs.random_cloud(6, CB, CP)
    cx, cy = torch.from_numpy(cx_h).to(device), torch.from_numpy(cy_h).to(device)
    ms = _timed(lambda: pc.pc_chamfer(cx, cy), steps, warm, flush, stream)
    pairs = 2.0 * CB * CP * CP
    tfl = pairs * FLOPS_PER_PAIR / (ms / 1e3) / 1e12
    out["chamfer"] = {
        "workload": f"B={CB}, P1=P2={CP} uniform in [0,1)^3, bidirectional, point+batch mean",
        "ms": ms, "clouds_per_s": CB * world / (ms / 1e3),
        "pairs": pairs, "achieved_tflops": tfl,
        "roofline": {"bound": "alu", "achieved": tfl, "peak": alu, "unit": "TFLOP/s",
                     "frac": tfl / alu}, "launches": 3}

    # three_interpolate forward / backward at the PointNet++ FP shape
    TB, TM, TN, TC = 16, 1024, 4096, 256
    px_h = inputs.pointnet2()                       # [16, 4096, 3]
    px = torch.from_numpy(px_h).to(device)
    centers = torch.from_numpy(np.ascontiguousarray(px_h[:, :TM])).to(device)
    d, idx = pc.three_nn(px, centers)
    w = 1.0 / (d + 1e-8)
    w = (w / w.sum(-1, keepdim=True)).contiguous()
    feats = torch.randn((TB, TC, TM), generator=torch.Generator(device="cpu").manual_seed(7)).to(device)
    g = torch.randn((TB, TC, TN), generator=torch.Generator(device="cpu").manual_seed(8)).to(device)
    fout = torch.empty((TB, TC, TN), dtype=torch.float32, device=device)
    gout = torch.empty((TB, TC, TM), dtype=torch.float32, device=device)
    fwd = _timed(lambda: pc.pc_three_interpolate(feats, idx, w, out=fout), steps, warm,
                 flush, stream)
    bwd = _timed(lambda: pc.pc_three_interpolate_backward(g, idx, w, TM, out=gout),
                 steps, warm, flush, stream)
    trip = TB * TN * 3 * (8 + 4)
    fwd_bytes = 4.0 * TB * TC * TN + 4.0 * TB * TC * TM + trip
    bwd_bytes = 4.0 * TB * TC * TN + 4.0 * TB * TC * TM + trip
    out["three_interpolate"] = {
        "workload": f"B={TB}, M={TM} centers -> n={TN} points, C={TC} channels, "
                    "indices from three_nn, inverse-distance weights",
        "forward_ms": fwd, "backward_ms": bwd,
        "forward_algorithmic_bytes": fwd_bytes, "backward_algorithmic_bytes": bwd_bytes,
        "forward_roofline": {"bound": "hbm", "achieved": fwd_bytes / (fwd / 1e3) / 1e9,
                             "peak": hbm, "unit": "GB/s",
                             "frac": fwd_bytes / (fwd / 1e3) / 1e9 / hbm},
        "backward_roofline": {"bound": "hbm", "achieved": bwd_bytes / (bwd / 1e3) / 1e9,
                              "peak": hbm, "unit": "GB/s",
                              "frac": bwd_bytes / (bwd / 1e3) / 1e9 / hbm},
        "launches": {"forward": 1,
                     "backward": "3 (entry lists, segment sort, ordered sums)"}}

    # PyTorch3D-style Ball Query with return_nn
    bq_ms = _timed(lambda: p3d_ball_query(centers, px, K=64, radius=0.2), steps, warm,
                   flush, stream)
    out["pytorch3d_ball_query"] = {
        "workload": f"B={TB}, {TM} centers vs {TN} points, r=0.2, K=64, return_nn",
        "ms": bq_ms, "queries_per_s": TB * TM * world / (bq_ms / 1e3), "launches": 2}

    # FPS at 1M points (workload 5: 16384 samples), the cooperative-grid
    # schedule (too large for one cluster)
    vx_h = inputs.very_large()
    vx = torch.from_numpy(vx_h).to(device)
    fps_out_v = torch.empty((1, 16384), dtype=torch.int64, device=device)
    ws_v = torch.empty(max(pc.binding.lib().pc_fps_workspace_bytes(1, vx_h.shape[1], 16384),
                           256), dtype=torch.uint8, device=device)
    fv_ms = _timed(lambda: pc.pc_fps(vx, 16384, 0, out=fps_out_v, workspace=ws_v),
                   max(3, min(steps, 5)), 3, flush, stream)
    out["fps_1m"] = {
        "workload": "N=1,000,000 uniform in [0,1)^3 with 1% duplicates, 16384 samples",
        "samples_per_s": 16384 * world / (fv_ms / 1e3), "launches": 1}
    out["fps_1m"].update(_fps_bounds(pc, vx_h.shape, 16384, fv_ms, device, flush, stream,
                                     float(peaks.get("sm_max_mhz", 2070.0)),
                                     max(3, min(steps, 5))))
    del vx, ws_v

    # kNN in D dimensions at the DGCNN EdgeConv feature shape
    DB, DN, DD, Dk = 32, 1024, 64, 20
    fx_h = np.random.default_rng(9).standard_normal((DB, DN, DD)).astype(np.float32)
    fx = torch.from_numpy(fx_h).to(device)
    kd_ms = _timed(lambda: pc.pc_knn_d(fx, fx, Dk), steps, warm, flush, stream)
    kd_flops = 3.0 * DD * DB * DN * DN
    kd_tfl = kd_flops / (kd_ms / 1e3) / 1e12
    out["knn_d"] = {
        "workload": f"B={DB} clouds of {DN} points with {DD}-d features, k={Dk}, "
                    "every point a query (DGCNN EdgeConv shape)",
        "ms": kd_ms, "queries_per_s": DB * DN * world / (kd_ms / 1e3),
        "algorithmic_flops": kd_flops,
        "roofline": {"bound": "alu", "achieved": kd_tfl, "peak": alu,
                     "unit": "TFLOP/s", "frac": kd_tfl / alu,
                     "note": "3 flops (sub, mul, add) per dimension and pair"},
        "launches": 1}

    if with_oracle:
        import oracle
        threads = os.cpu_count() or 1
        krows = np.arange(0, DB * DN, DB * DN // (16 * threads), dtype=np.int64)
        t0 = time.perf_counter()
        oracle.knn_d(fx_h, fx_h, Dk, rows=krows, threads=threads)
        t1 = time.perf_counter()
        out["knn_d"]["oracle"] = {
            "ms_extrapolated": (t1 - t0) / len(krows) * DB * DN * 1e3,
            "cores": threads, "sample": f"{len(krows)} query rows, extrapolated"}
        rows = np.arange(0, CB * CP, CB * CP // (64 * threads), dtype=np.int64)
        t0 = time.perf_counter()
        oracle.knn_masked(cx_h, cy_h, 1, squared=True, rows=rows, threads=threads)
        t1 = time.perf_counter()
        per_row = (t1 - t0) / len(rows)
        out["chamfer"]["oracle"] = {
            "ms_extrapolated": per_row * 2 * CB * CP * 1e3, "cores": threads,
            "sample": f"{len(rows)} nearest-neighbour rows of one direction, "
                      "extrapolated to both directions"}
        fi, ii, wi = feats.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()
        t0 = time.perf_counter()
        oracle.three_interpolate(fi, ii, wi)
        t1 = time.perf_counter()
        oracle.three_interpolate_backward(g.cpu().numpy(), ii, wi, TM)
        t2 = time.perf_counter()
        out["three_interpolate"]["oracle"] = {
            "forward_ms": (t1 - t0) * 1e3, "backward_ms": (t2 - t1) * 1e3, "cores": 1,
            "sample": "full workload, single thread"}
        qrows = np.arange(0, TB * TM, 16, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.ball_query_masked(np.ascontiguousarray(px_h[:, :TM]), px_h, 0.2, 64,
                                 rows=qrows)
        t1 = time.perf_counter()
        out["pytorch3d_ball_query"]["oracle"] = {
            "ms_extrapolated": (t1 - t0) / len(qrows) * TB * TM * 1e3, "cores": 1,
            "sample": f"{len(qrows)} query rows (gather not included), extrapolated"}
    return out


# ---------------------------------------------------------------------------
# every workload: FPS, kNN and Ball Query of each configuration, timed alone
# ---------------------------------------------------------------------------
FPS_INSTR_PER_POINT_STEP = 10   # min update, compare and select per point-step


def _fps_bounds(pc, x_shape, npoint, ms, device, flush, stream, max_mhz, steps):
    """FPS against the bounds it does face: the ALU work on the SMs its
    schedule holds, and the measured floor of its per-step reduction and
    exchange (the same schedule, same sample count, 1024 points per block)."""
    import torch
    from point_cloud_neighbor_gb300 import inputs
    B, N = int(x_shape[0]), int(x_shape[1])
    strategy, cs, bpc = pc.pc_fps_plan(B, N)
    sms = pc.pc_fps_sm_count(B, N, npoint)
    alu_ms = (float(B) * N * (npoint - 1) * FPS_INSTR_PER_POINT_STEP /
              (max(sms, 1) * 128 * max_mhz * 1e6) * 1e3)
    n_floor = 1024 * bpc
    fx = torch.from_numpy(inputs.random_cloud(7, B, n_floor)).to(device)
    kw = {"strategy": strategy}
    if strategy == pc.PC_FPS_CLUSTER:
        kw["cluster_size"] = bpc
    elif strategy == pc.PC_FPS_GRID:
        kw["blocks_per_cloud"] = bpc
        kw["cluster_size"] = cs
    try:
        floor_ms = _timed(lambda: pc.pc_fps(fx, npoint, 0, **kw), steps, 3, flush, stream)
    except pc.PointCloudError as err:
        floor_ms = None
        note = f"floor not measured: {err}"
    else:
        note = (f"the same schedule on {n_floor} points per cloud "
                f"(1024 per block), npoint={npoint}")
    names = {pc.PC_FPS_BLOCK: "block", pc.PC_FPS_CLUSTER: "cluster",
             pc.PC_FPS_GRID: "grid"}
    out = {"schedule": names.get(strategy, str(strategy)), "cluster_size": cs,
           "blocks_per_cloud": bpc,
           "sms": sms, "ms": ms, "us_per_step": ms * 1e3 / max(npoint - 1, 1),
           "alu_bound_ms": alu_ms, "alu_frac": alu_ms / ms,
           "floor_ms": floor_ms, "floor_frac": (floor_ms / ms) if floor_ms else None,
           "floor_note": note,
           "streamed_equivalent_gbs": float(B) * N * (npoint - 1) *
           FPS_BYTES_PER_POINT_STEP / (ms / 1e3) / 1e9}
    out["roofline"] = {
        "bound": "latency", "achieved": out["us_per_step"],
        "peak": (floor_ms * 1e3 / max(npoint - 1, 1)) if floor_ms else None,
        "unit": "us per step", "frac": out["floor_frac"],
        "note": "measured floor of the schedule's per-step reduction and exchange "
                "(the kernel keeps points and minima on chip: no HBM stream)"}
    return out


def _oracle_timing(fn, units, budget_s):
    """Seconds per unit of one oracle call on a bounded sample: fn(n) runs the
    oracle on n units; n doubles from 1 until a call takes budget_s / 4."""
    n = 1
    while True:
        t0 = time.perf_counter()
        fn(n)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or n >= units:
            return dt / n, n
        n = min(units, n * max(2, int(budget_s / 4 / max(dt, 1e-4))))


def run_configs(args, pc, flush, device, world, with_oracle):
    """The five workloads, each operator timed alone (CUDA events on the
    launching stream, L2 flushed before every call), with its roofline
    fraction and, on rank 0, the oracle timed on the host cores single-threaded
    and on all cores (bounded samples, extrapolated per unit)."""
    import torch
    from point_cloud_neighbor_gb300 import inputs
    stream = torch.cuda.current_stream(device)
    steps, warm = max(3, min(args.steps, 10)), 3
    peaks, peak_kind = measured_peaks()
    max_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    alu = fp32_alu_peak_tflops(sm_count, max_mhz)
    threads = os.cpu_count() or 1
    if with_oracle:
        import oracle
        oracle.build()
    out = {}
    plan = [
        ("tiny", "tiny", False),
        ("point_mae", "point_mae", False),
        ("pointnet2", "pointnet2", False),
        ("large_morton", "large", True),
        ("very_large", "very_large", False),
    ]
    for name, base, morton in plan:
        cfg = inputs.CONFIGS[base]
        xh = inputs.large(morton=True) if morton else inputs.make(base)
        x = torch.from_numpy(xh).to(device)
        B, N = xh.shape[0], xh.shape[1]
        npoint = cfg["npoint"]
        entry = {"B": B, "N": N}
        fo = torch.empty((B, npoint), dtype=torch.int64, device=device)
        ms = _timed(lambda: pc.pc_fps(x, npoint, 0, out=fo), steps, warm, flush, stream)
        fps = {"npoint": npoint, "samples_per_s": B * npoint * world / (ms / 1e3)}
        fps.update(_fps_bounds(pc, xh.shape, npoint, ms, device, flush, stream,
                               max_mhz, steps))
        entry["fps"] = fps
        cen = torch.gather(x, 1, fo.unsqueeze(-1).expand(B, npoint, 3)).contiguous()
        centers_h = cen.cpu().numpy()
        # kNN: queries and references of the workload
        k = cfg["knn_k"]
        if name == "pointnet2":          # three_nn shape: points vs centres
            kq, kr, kq_h, kr_h = x, cen, xh, centers_h
        elif name == "large_morton":     # every point a query
            kq, kr, kq_h, kr_h = x, x, xh, xh
        else:                            # the FPS centres as queries
            kq, kr, kq_h, kr_h = cen, x, centers_h, xh
        Q, Nr = kq.shape[1], kr.shape[1]
        kd = torch.empty((B, Q, k), dtype=torch.float32, device=device)
        ki = torch.empty((B, Q, k), dtype=torch.int64, device=device)
        ms = _timed(lambda: pc.pc_knn(kq, kr, k, out_dist=kd, out_idx=ki), steps, warm,
                    flush, stream)
        pairs = float(B) * Q * Nr
        tfl = pairs * FLOPS_PER_PAIR / (ms / 1e3) / 1e12
        entry["knn"] = {"k": k, "queries": B * Q, "references_per_cloud": Nr, "ms": ms,
                        "queries_per_s": B * Q * world / (ms / 1e3), "pairs": pairs,
                        "roofline": {"bound": "alu", "achieved": tfl, "peak": alu,
                                     "unit": "TFLOP/s", "frac": tfl / alu}}
        if with_oracle:
            rows_total = B * Q
            rng = np.random.default_rng(11)
            perm = rng.permutation(rows_total).astype(np.int64)
            per1, n1 = _oracle_timing(
                lambda n: oracle.knn(kq_h, kr_h, k, rows=np.sort(perm[:n])),
                rows_total, 2.0)
            perT, nT = _oracle_timing(
                lambda n: oracle.knn(kq_h, kr_h, k, rows=np.sort(perm[:n]), threads=threads),
                rows_total, 2.0)
            entry["knn"]["oracle"] = {
                "single_thread_ms": per1 * rows_total * 1e3,
                "all_cores_ms": perT * rows_total * 1e3, "cores": threads,
                "sample": f"{n1} rows on 1 thread, {nT} rows on {threads}, "
                          "extrapolated to all rows"}
        # Ball Query: the workload's radii on the FPS centres (every point
        # a query on the 100k cloud)
        bqs = []
        for r, K in cfg["bq"]:
            bq_q, bq_q_h = (x, xh) if name == "large_morton" else (cen, centers_h)
            Qb = bq_q.shape[1]
            bd = torch.empty((B, Qb, K), dtype=torch.float32, device=device)
            bi = torch.empty((B, Qb, K), dtype=torch.int64, device=device)
            ms = _timed(lambda: pc.pc_ball_query(bq_q, x, r, K, out_dist2=bd, out_idx=bi),
                        steps, warm, flush, stream)
            last = bi.cpu().numpy().reshape(-1, K)[:, K - 1]
            bpairs = float(np.where(last >= 0, last + 1, N).sum())
            tfl = bpairs * FLOPS_PER_PAIR / (ms / 1e3) / 1e12
            e = {"radius": r, "K": K, "queries": B * Qb, "ms": ms,
                 "queries_per_s": B * Qb * world / (ms / 1e3), "pairs": bpairs,
                 "roofline": {"bound": "alu", "achieved": tfl, "peak": alu,
                              "unit": "TFLOP/s", "frac": tfl / alu}}
            if with_oracle:
                rows_total = B * Qb
                perm = np.random.default_rng(12).permutation(rows_total).astype(np.int64)
                per1, n1 = _oracle_timing(
                    lambda n: oracle.ball_query(bq_q_h, xh, r, K, rows=np.sort(perm[:n])),
                    rows_total, 2.0)
                perT, nT = _oracle_timing(
                    lambda n: oracle.ball_query(bq_q_h, xh, r, K, rows=np.sort(perm[:n]),
                                                threads=threads),
                    rows_total, 2.0)
                e["oracle"] = {"single_thread_ms": per1 * rows_total * 1e3,
                               "all_cores_ms": perT * rows_total * 1e3, "cores": threads,
                               "sample": f"{n1} rows on 1 thread, {nT} rows on {threads}, "
                                         "extrapolated to all rows"}
            bqs.append(e)
        if bqs:
            entry["ball_query"] = bqs
        if with_oracle:
            # FPS: the first few samples of every cloud, extrapolated per sample
            def fps1(n, xh=xh):
                oracle.fps(xh, n + 1, 0)

            # all cores: several clouds run in parallel, one cloud's steps
            # split their points over the threads
            def fpsT(n, xh=xh):
                if B > 1:
                    oracle.fps(xh, n + 1, 0, threads=threads)
                else:
                    oracle.fps_all_cores(xh, n + 1, 0, threads=threads)
            per1, n1 = _oracle_timing(fps1, npoint - 1, 2.0)
            perT, nT = _oracle_timing(fpsT, npoint - 1, 2.0)
            how = (f"the {B} clouds over {threads} threads" if B > 1 else
                   f"each step's points split over {threads} threads")
            fps["oracle"] = {
                "single_thread_ms": per1 * (npoint - 1) * 1e3,
                "all_cores_ms": perT * (npoint - 1) * 1e3, "cores": threads,
                "sample": f"{n1} samples on 1 thread, {nT} samples with {how}, "
                          f"extrapolated to {npoint - 1} samples"}
        out[name] = entry
        del x
    return out


def run_e2e(args, pc, x_host, device, world, bq_first=True):
    """Same step through the public API with host buffers: the input is copied
    from pinned host memory each step and every result is read back into
    pinned host memory; wall time around each synchronized step.  Fused, the
    kNN and Ball Query results are read back on a copy stream as soon as
    their call ends, while FPS may still run.  Separate (--separate), with
    bq_first the side stream runs Ball Query before kNN, so that the larger
    read-back (Ball Query's K = 32 slots per query) overlaps kNN and only
    kNN's follows the last kernel."""
    import torch
    W = WORKLOAD
    N, npoint, k, r, K = W["N"], W["npoint"], W["knn_k"], W["bq_radius"], W["bq_K"]
    x_pin = torch.from_numpy(x_host).pin_memory()
    outs = {
        "fps": torch.empty((1, npoint), dtype=torch.int64).pin_memory(),
        "knn_d": torch.empty((1, N, k), dtype=torch.float32).pin_memory(),
        "knn_i": torch.empty((1, N, k), dtype=torch.int64).pin_memory(),
        "bq_d": torch.empty((1, N, K), dtype=torch.float32).pin_memory(),
        "bq_i": torch.empty((1, N, K), dtype=torch.int64).pin_memory(),
    }
    h2d = x_pin.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in outs.values())

    main = torch.cuda.current_stream(device)
    side = torch.cuda.Stream(device) if not args.serial else main
    # the first operator's results are read back while the second runs, the
    # FPS result once FPS ends; only the second's read-back follows the last
    # kernel
    copy = torch.cuda.Stream(device) if not args.serial else main
    reserve = 0 if args.serial else args.fps_cluster

    def one_fused():
        xd = x_pin.to(device, non_blocking=True)
        side.wait_stream(main)
        f = pc.pc_fps(xd, npoint, 0, strategy=pc.PC_FPS_CLUSTER,
                      cluster_size=args.fps_cluster)
        outs["fps"].copy_(f, non_blocking=True)
        with torch.cuda.stream(side):
            pc.pc_set_sm_reserve(reserve)
            res = pc.pc_knn_ball_query(xd, xd, k, r, K)
            pc.pc_set_sm_reserve(0)
        copy.wait_stream(side)
        with torch.cuda.stream(copy):
            for t, name in zip(res, ("knn_d", "knn_i", "bq_d", "bq_i")):
                t.record_stream(copy)
                outs[name].copy_(t, non_blocking=True)
        torch.cuda.synchronize(device)

    def one():
        if not args.separate:
            one_fused()
            return
        xd = x_pin.to(device, non_blocking=True)
        side.wait_stream(main)
        f = pc.pc_fps(xd, npoint, 0, strategy=pc.PC_FPS_CLUSTER,
                      cluster_size=args.fps_cluster)
        outs["fps"].copy_(f, non_blocking=True)
        ops = [("knn", lambda: pc.pc_knn(xd, xd, k)),
               ("bq", lambda: pc.pc_ball_query(xd, xd, r, K))]
        if bq_first:
            ops.reverse()
        with torch.cuda.stream(side):
            pc.pc_set_sm_reserve(reserve)
            first = ops[0][1]()
            copy.wait_stream(side)
            second = ops[1][1]()
            pc.pc_set_sm_reserve(0)
        names = {"knn": ("knn_d", "knn_i"), "bq": ("bq_d", "bq_i")}
        with torch.cuda.stream(copy):
            for t, name in zip(first, names[ops[0][0]]):
                t.record_stream(copy)
                outs[name].copy_(t, non_blocking=True)
        main.wait_stream(side)
        for t, name in zip(second, names[ops[1][0]]):
            t.record_stream(main)
            outs[name].copy_(t, non_blocking=True)
        torch.cuda.synchronize(device)

    for _ in range(max(1, args.warmup)):
        one()
    steps = max(3, min(args.steps, 20))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    t1 = time.perf_counter()
    (elapsed,) = max_over_ranks([t1 - t0], world, device)
    value = (N + N) * world * steps / elapsed
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": elapsed / steps * 1e3,
            "note": "pinned host input copied in and all outputs read back every step",
            "knn_ball_query": "pc_knn then pc_ball_query" if args.separate else "one fused call"}


# ---------------------------------------------------------------------------
# CPU oracle timings (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step_costs(x_host, knn_rows, bq_rows, fps_steps, threads, seed=0):
    """Seconds per kNN query, per Ball Query query and per FPS sample of the
    oracle, measured on bounded samples of the workload."""
    import oracle
    oracle.build()
    W = WORKLOAD
    N = W["N"]
    rng = np.random.default_rng(seed)
    rk = np.sort(rng.choice(N, knn_rows, replace=False)).astype(np.int64)
    rb = np.sort(rng.choice(N, bq_rows, replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    oracle.knn(x_host, x_host, W["knn_k"], rows=rk, threads=threads)
    t1 = time.perf_counter()
    oracle.ball_query(x_host, x_host, W["bq_radius"], W["bq_K"], rows=rb,
                      threads=threads)
    t2 = time.perf_counter()
    if threads > 1:       # each step's points split over the threads
        oracle.fps_all_cores(x_host, fps_steps + 1, 0, threads=threads)
    else:
        oracle.fps(x_host, fps_steps + 1, 0)
    t3 = time.perf_counter()
    return {"knn_s_per_query": (t1 - t0) / knn_rows,
            "bq_s_per_query": (t2 - t1) / bq_rows,
            "fps_s_per_sample": (t3 - t2) / fps_steps,
            "knn_rows": knn_rows, "bq_rows": bq_rows, "fps_steps": fps_steps,
            "elapsed_s": t3 - t0}


def extrapolated_step_s(c):
    W = WORKLOAD
    return (c["knn_s_per_query"] * W["N"] + c["bq_s_per_query"] * W["N"] +
            c["fps_s_per_sample"] * (W["npoint"] - 1))


def cpu_baseline(x_host, budget_s=20.0):
    threads = os.cpu_count() or 1
    # calibrate sample sizes so the whole leg takes about budget_s
    probe = oracle_step_costs(x_host, knn_rows=threads, bq_rows=16 * threads,
                              fps_steps=16, threads=threads)
    share = budget_s / 3.0
    knn_rows = int(max(threads, min(4096, share / max(probe["knn_s_per_query"], 1e-9))))
    bq_rows = int(max(threads, min(100000, share / max(probe["bq_s_per_query"], 1e-9))))
    fps_steps = int(max(8, min(4095, share / max(probe["fps_s_per_sample"], 1e-9))))
    c = oracle_step_costs(x_host, knn_rows, bq_rows, fps_steps, threads, seed=1)
    step_s = extrapolated_step_s(c)
    # the same oracle on one thread (smaller samples)
    one = oracle_step_costs(x_host, max(2, knn_rows // (2 * threads)),
                            max(16, bq_rows // (2 * threads)), max(8, fps_steps // 4),
                            1, seed=2)
    step1_s = extrapolated_step_s(one)
    return {"value": 2 * WORKLOAD["N"] / step_s, "unit": UNIT, "cores": threads,
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": (f"{knn_rows} kNN queries and {bq_rows} Ball Query queries "
                       f"on {threads} threads, {fps_steps} FPS samples with each "
                       f"step's points split over {threads} threads, extrapolated "
                       f"to the full step"),
            "step_s_extrapolated": step_s, "measured_s": c["elapsed_s"],
            "per_unit_s": {k: c[k] for k in ("knn_s_per_query", "bq_s_per_query",
                                             "fps_s_per_sample")},
            "single_thread": {
                "value": 2 * WORKLOAD["N"] / step1_s, "step_s_extrapolated": step1_s,
                "sample": (f"{one['knn_rows']} kNN queries, {one['bq_rows']} Ball Query "
                           f"queries and {one['fps_steps']} FPS samples on 1 thread, "
                           f"extrapolated to the full step"),
                "per_unit_s": {k: one[k] for k in ("knn_s_per_query", "bq_s_per_query",
                                                   "fps_s_per_sample")}}}


ARM_PARTS = {(0x41, 0xd4f): "Arm Neoverse V2", (0x41, 0xd40): "Arm Neoverse V1",
             (0x41, 0xd0c): "Arm Neoverse N1", (0x41, 0xd8e): "Arm Neoverse N3",
             (0x41, 0xd84): "Arm Neoverse V3"}


def cpu_model() -> str:
    """The host CPU's model name from /proc/cpuinfo ("model name" on x86;
    the implementer and part numbers on Arm), else the architecture."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    key, val = line.split(":", 1)
                    fields.setdefault(key.strip().lower(), val.strip())
    except OSError:
        return platform.machine()
    for key in ("model name", "cpu model", "hardware"):
        if fields.get(key):
            return fields[key]
    try:
        impl = int(fields["cpu implementer"], 16)
        part = int(fields["cpu part"], 16)
    except (KeyError, ValueError):
        return platform.machine()
    return ARM_PARTS.get((impl, part),
                         f"{platform.machine()} implementer {impl:#x} part {part:#x}")


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return   # the CPU oracle runs once, on rank 0
    from point_cloud_neighbor_gb300 import inputs
    x_host = inputs.large(seed=3, morton=False)
    threads = os.cpu_count() or 1
    knn_rows, bq_rows, fps_steps = 2 * threads, 64 * threads, 16
    for _ in range(args.warmup):
        oracle_step_costs(x_host, knn_rows, bq_rows, fps_steps, threads, seed=99)
    costs = [oracle_step_costs(x_host, knn_rows, bq_rows, fps_steps, threads,
                               seed=s) for s in range(args.steps)]
    agg = {k: statistics.mean(c[k] for c in costs)
           for k in ("knn_s_per_query", "bq_s_per_query", "fps_s_per_sample")}
    step_s = extrapolated_step_s(agg)
    value = 2 * WORKLOAD["N"] / step_s
    sample = (f"per step {knn_rows} kNN queries and {bq_rows} Ball Query queries "
              f"on {threads} threads and {fps_steps} FPS samples with each step's "
              f"points split over {threads} threads, extrapolated to the full step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config({"parallelism": "host cores, oracle"}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        "per_unit_s": agg,
    }))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle work for the cpu_baseline leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step-only", action="store_true",
                    help="time only the FPS + kNN + Ball Query step (no grid, "
                         "next-row or end-to-end sections; for profiler captures)")
    ap.add_argument("--fps-cluster", type=int, default=STEP_FPS_CLUSTER,
                    help="blocks of the FPS cluster in the step (its SMs are "
                         "reserved from the kNN + Ball Query grid)")
    ap.add_argument("--separate", action="store_true",
                    help="run kNN and Ball Query of the step as two calls "
                         "(pc_knn, pc_ball_query) instead of one fused call")
    ap.add_argument("--serial", action="store_true",
                    help="run FPS, kNN and Ball Query one after another on one "
                         "stream instead of FPS concurrently on a side stream")
    ap.add_argument("--only", choices=["fps", "knn", "ball_query", "knn_ball_query",
                                       "grid_build",
                                       "grid_knn", "grid_ball_query", "chamfer",
                                       "three_interpolate",
                                       "three_interpolate_backward", "knn_d",
                                       "fps_1m", "knn_1m", "ball_query_1m"],
                    help="run one operator of the step W + K times and print "
                         "its mean CUDA-event time (for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
