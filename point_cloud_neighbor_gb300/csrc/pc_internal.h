// pc_internal.h -- host-side declarations shared by the launchers and the C
// ABI (not installed; the public interface is include/pointcloud.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pcn {

// Cached properties of one device, filled once per device.
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    int warp_size = 0;
    size_t smem_per_block_optin = 0;
    size_t smem_per_sm = 0;
    int max_threads_per_sm = 0;
    int cooperative = 0;
    int *status_word = nullptr;  // device address of the status word
    // the library's stream-ordered pool for kernel scratch (nullptr: the
    // device's default pool)
    cudaMemPool_t scratch_pool = nullptr;
};

// Scratch memory for the library's own kernels, stream-ordered on `stream`:
// from the device's library pool, which keeps up to 256 MiB reserved
// between calls (the default pool returns freed memory at every
// synchronization, so a caller that synchronizes after each call would pay
// for mapping it again on every call).
cudaError_t scratch_alloc(const DeviceInfo &dev, void **p, size_t bytes,
                          cudaStream_t stream);
cudaError_t scratch_free(void *p, cudaStream_t stream);

// Device-side wait bound, in ns (see pc_set_wait_timeout_ns).
uint64_t wait_timeout_ns();
// SMs taken by concurrent work (see pc_set_sm_reserve).
int sm_reserve();
// Testing hooks: the PC_STALL_* flags set by pc_debug_set_stall.
int debug_stall();

// Device resolution, pointer checks and error messages of the C ABI, for
// entry points defined outside pc_api.cu.
int api_current_device(const DeviceInfo **out);
int api_check_ptr(const void *p, int dev, size_t align, const char *name);
int api_fail(int code, const char *message);

// Launch plans --------------------------------------------------------------
struct ScanPlan {       // kNN / Ball Query
    int warps = 8;      // warps per block
    int q_per_warp = 1; // queries per warp
    int blocks_per_cloud = 1;
    int ntiles = 0;     // reference tiles per cloud
    int tile_stride = 1;
    size_t smem_bytes = 0;
};

// Launchers: enqueue on `stream`, return the first CUDA error.
// q_len / r_len: valid queries / references per cloud (device, NULL = all);
// rows past q_len and slots past r_len are padded with (-1, 0).
cudaError_t launch_knn(const DeviceInfo &dev, const float *query, int64_t B,
                       int64_t Q, const float *ref, int64_t N, int k,
                       const int64_t *q_len, const int64_t *r_len, bool squared,
                       float *out_dist, int64_t *out_idx, cudaStream_t stream);

// Two kNN problems with the same B and k in one launch when k <= 32 (the
// Chamfer distance's two directions); two launches otherwise.
cudaError_t launch_knn_pair(const DeviceInfo &dev, int64_t B, int k, bool squared,
                            const float *q0, int64_t Q0, const float *r0, int64_t N0,
                            const int64_t *ql0, const int64_t *rl0, float *d0,
                            int64_t *i0, const float *q1, int64_t Q1,
                            const float *r1, int64_t N1, const int64_t *ql1,
                            const int64_t *rl1, float *d1, int64_t *i1,
                            cudaStream_t stream);

cudaError_t launch_ball_query(const DeviceInfo &dev, const float *query,
                              int64_t B, int64_t Q, const float *ref,
                              int64_t N, const int64_t *q_len,
                              const int64_t *r_len, float r32, int64_t K,
                              float *out_dist2, int64_t *out_idx,
                              cudaStream_t stream);

// kNN and Ball Query of the same queries against the same references; one
// fused launch where knn_ball_query_fused holds, else launch_knn then
// launch_ball_query.  No lengths; kNN distances are sqrt(s).
bool knn_ball_query_fused(const DeviceInfo &dev, int64_t B, int64_t Q, int64_t N,
                          int k, float r32, int64_t K);
cudaError_t launch_knn_ball_query(const DeviceInfo &dev, const float *query, int64_t B,
                                  int64_t Q, const float *ref, int64_t N, int k,
                                  float *knn_dist, int64_t *knn_idx, float r32, int64_t K,
                                  float *bq_dist2, int64_t *bq_idx, cudaStream_t stream);

// FPS of the CLUSTER schedule in rounds of several centers per exchange: 1
// (default) or 0 = one center per exchange (pc_fps_set_batched).
int fps_batched();

struct FpsPlan {
    int strategy = 0;       // PC_FPS_BLOCK / CLUSTER / GRID
    int cluster = 1;        // blocks per cluster (BLOCK: 1)
    int blocks_per_cloud = 1;
    int threads = 1024;
    int ppt = 1;            // points per thread
    int chunk = 0;          // points per block
    size_t smem_bytes = 0;
    size_t workspace_bytes = 0;
    // two-level GRID: the rounds kernel fits (threads with its resolving
    // warp, its shared memory); workspace_bytes then covers it, and
    // step_workspace_bytes is what the step-by-step kernel alone needs
    bool grid_rounds = false;
    int rounds_ppt = 0;
    int rounds_threads = 0;
    size_t rounds_smem = 0;
    size_t step_workspace_bytes = 0;
    bool ok = false;
    const char *why = "";
};

FpsPlan plan_fps(const DeviceInfo &dev, int64_t B, int64_t N, int strategy,
                 int cluster_size, int blocks_per_cloud);

cudaError_t launch_fps(const DeviceInfo &dev, const FpsPlan &plan,
                       const float *xyz, int64_t B, int64_t N, int64_t npoint,
                       int64_t start_idx, int64_t *out_idx, void *workspace,
                       cudaStream_t stream);

}  // namespace pcn
