// pc_api.cu -- the C ABI of libpointcloud.so (declared in
// include/pointcloud.h): host-side validation, device checks, schedule
// choice, workspace handling and the device status word.  Every compute step
// runs in the kernels of pc_fps.cu, pc_knn.cu and pc_ball_query.cu.
#include "pointcloud.h"
#include "pc_internal.h"

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

namespace {

// The device status word: the first device-side error (a bounded wait that
// ran out) is recorded here.  One instance per device (module global).
__device__ int g_device_status = 0;

constexpr int kMaxDevices = 64;
constexpr int kVersion = 10000 * 0 + 100 * 1 + 0;  // 0.1.0

thread_local std::string t_error;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_sm_reserve{0};
std::atomic<int> g_fps_batched{1};
std::atomic<int> g_stall{0};  // PC_STALL_* testing flags
std::mutex g_dev_mutex;
pcn::DeviceInfo g_devices[kMaxDevices];
bool g_device_ready[kMaxDevices] = {};

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(PC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                cudaGetErrorString(e));
}

// Resolve and cache the current device; checks that it is the architecture
// this library is built for (compute capability 10.3, 32-wide warps).
int current_device(const pcn::DeviceInfo **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PC_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PC_ERR_NO_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_device_ready[dev]) {
        pcn::DeviceInfo d;
        d.device = dev;
        int v = 0;
        auto attr = [&](cudaDeviceAttr a) {
            v = 0;
            cudaDeviceGetAttribute(&v, a, dev);
            return v;
        };
        d.sm_count = attr(cudaDevAttrMultiProcessorCount);
        d.cc_major = attr(cudaDevAttrComputeCapabilityMajor);
        d.cc_minor = attr(cudaDevAttrComputeCapabilityMinor);
        d.warp_size = attr(cudaDevAttrWarpSize);
        d.smem_per_block_optin = size_t(attr(cudaDevAttrMaxSharedMemoryPerBlockOptin));
        d.smem_per_sm = size_t(attr(cudaDevAttrMaxSharedMemoryPerMultiprocessor));
        d.max_threads_per_sm = attr(cudaDevAttrMaxThreadsPerMultiProcessor);
        d.cooperative = attr(cudaDevAttrCooperativeLaunch);
        if (d.cc_major != 10 || d.cc_minor != 3)
            return fail(PC_ERR_NO_DEVICE,
                        "device %d has compute capability %d.%d; this library "
                        "is built for sm_103a only", dev, d.cc_major, d.cc_minor);
        if (d.warp_size != 32)
            return fail(PC_ERR_NO_DEVICE, "device %d reports warp size %d, need 32",
                        dev, d.warp_size);
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) return cuda_fail(e, "status word address");
        d.status_word = static_cast<int *>(p);
        // the scratch pool: device memory, kept up to 256 MiB between calls;
        // without it (pools unsupported) scratch comes from the default pool
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
            uint64_t keep = uint64_t(256) << 20;
            if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) ==
                cudaSuccess)
                d.scratch_pool = pool;
            else
                cudaMemPoolDestroy(pool);
        }
        cudaGetLastError();
        g_devices[dev] = d;
        g_device_ready[dev] = true;
    }
    *out = &g_devices[dev];
    return PC_OK;
}

// A caller pointer must be device (or managed) memory of `dev`, aligned.
int check_ptr(const void *p, int dev, size_t align, const char *name) {
    if (p == nullptr) return fail(PC_ERR_INVALID_ARGUMENT, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) % align != 0)
        return fail(PC_ERR_INVALID_ARGUMENT, "%s is not %zu-byte aligned", name,
                    align);
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(PC_ERR_INVALID_ARGUMENT, "%s is not a CUDA pointer (%s)",
                    name, cudaGetErrorString(e));
    }
    if (at.type == cudaMemoryTypeManaged) return PC_OK;
    if (at.type != cudaMemoryTypeDevice)
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "%s is not device memory (host pointers are not accepted)",
                    name);
    if (at.device != dev)
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "%s lives on device %d but device %d is current", name,
                    at.device, dev);
    return PC_OK;
}

constexpr int64_t kMaxInt = 2147483647;
constexpr int64_t kMaxElems = int64_t(1) << 62;

bool mul_ok(int64_t a, int64_t b, int64_t c) {
    if (a == 0 || b == 0 || c == 0) return true;
    return a <= kMaxElems / b && a * b <= kMaxElems / c;
}

}  // namespace

namespace pcn {
cudaError_t scratch_alloc(const DeviceInfo &dev, void **p, size_t bytes,
                          cudaStream_t stream) {
    if (dev.scratch_pool != nullptr)
        return cudaMallocFromPoolAsync(p, bytes, dev.scratch_pool, stream);
    return cudaMallocAsync(p, bytes, stream);
}
cudaError_t scratch_free(void *p, cudaStream_t stream) { return cudaFreeAsync(p, stream); }

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }
int sm_reserve() { return g_sm_reserve.load(); }
int fps_batched() { return g_fps_batched.load(); }
int debug_stall() { return g_stall.load(); }
int api_current_device(const DeviceInfo **out) { return current_device(out); }
int api_check_ptr(const void *p, int dev, size_t align, const char *name) {
    return check_ptr(p, dev, align, name);
}
int api_fail(int code, const char *message) { return fail(code, "%s", message); }
}  // namespace pcn

extern "C" {

const char *pc_status_string(int status) {
    switch (status) {
        case PC_OK: return "PC_OK";
        case PC_ERR_INVALID_ARGUMENT: return "PC_ERR_INVALID_ARGUMENT";
        case PC_ERR_UNSUPPORTED: return "PC_ERR_UNSUPPORTED";
        case PC_ERR_CUDA: return "PC_ERR_CUDA";
        case PC_ERR_DEVICE_TIMEOUT: return "PC_ERR_DEVICE_TIMEOUT";
        case PC_ERR_NO_DEVICE: return "PC_ERR_NO_DEVICE";
        default: return "PC_ERR_UNKNOWN";
    }
}

const char *pc_last_error_message(void) { return t_error.c_str(); }

int pc_version(void) { return kVersion; }

void pc_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns < 1000 ? 1000 : ns);
}

void pc_debug_set_fps_grid_stall(int enable) {
    if (enable)
        g_stall.fetch_or(PC_STALL_FPS_GRID);
    else
        g_stall.fetch_and(~PC_STALL_FPS_GRID);
}

void pc_debug_set_stall(int mask) {
    g_stall.store(mask & (PC_STALL_FPS_GRID | PC_STALL_FPS_CLUSTER | PC_STALL_TILE_STREAM));
}

void pc_set_sm_reserve(int sms) { g_sm_reserve.store(sms < 0 ? 0 : sms); }

int pc_fps_set_batched(int enable) { return g_fps_batched.exchange(enable ? 1 : 0); }

int pc_fps_sm_count(int64_t B, int64_t N, int64_t npoint) {
    (void)npoint;
    if (B <= 0 || N <= 0) return 0;
    const pcn::DeviceInfo *dev = nullptr;
    if (current_device(&dev) != PC_OK) return 0;
    const pcn::FpsPlan p = pcn::plan_fps(*dev, B, N, PC_FPS_AUTO, 0, 0);
    if (!p.ok) return 0;
    return int(std::min<int64_t>(dev->sm_count, B * int64_t(p.blocks_per_cloud)));
}

int pc_fps_plan(int64_t B, int64_t N, int strategy, int cluster_size,
                int blocks_per_cloud, int *out_strategy, int *out_cluster_size,
                int *out_blocks_per_cloud) {
    if (out_strategy == nullptr || out_cluster_size == nullptr ||
        out_blocks_per_cloud == nullptr)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, "fps_plan: null output pointer");
    *out_strategy = 0;
    *out_cluster_size = 0;
    *out_blocks_per_cloud = 0;
    if (B <= 0 || N <= 0)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, "fps_plan: need B > 0 and N > 0");
    const pcn::DeviceInfo *dev = nullptr;
    const int rc = current_device(&dev);
    if (rc != PC_OK) return rc;
    const pcn::FpsPlan p = pcn::plan_fps(*dev, B, N, strategy, cluster_size,
                                         blocks_per_cloud);
    if (!p.ok) {
        char msg[256];
        std::snprintf(msg, sizeof(msg), "fps_plan: %s", p.why);
        return pcn::api_fail(PC_ERR_UNSUPPORTED, msg);
    }
    *out_strategy = p.strategy;
    *out_cluster_size = p.cluster;
    *out_blocks_per_cloud = p.blocks_per_cloud;
    return PC_OK;
}

size_t pc_fps_workspace_bytes_ex(int64_t B, int64_t N, int64_t npoint,
                                 int strategy, int blocks_per_cloud) {
    (void)npoint;
    if (B <= 0 || N <= 0) return 0;
    const pcn::DeviceInfo *dev = nullptr;
    if (current_device(&dev) != PC_OK) return 0;
    pcn::FpsPlan p = pcn::plan_fps(*dev, B, N, strategy, 0, blocks_per_cloud);
    return p.ok ? p.workspace_bytes : 0;
}

size_t pc_fps_workspace_bytes(int64_t B, int64_t N, int64_t npoint) {
    return pc_fps_workspace_bytes_ex(B, N, npoint, PC_FPS_AUTO, 0);
}

int pc_fps_ex(const float *xyz, int64_t B, int64_t N, int64_t npoint,
              int64_t start_idx, int64_t *out_idx, void *workspace,
              size_t workspace_bytes, int strategy, int cluster_size,
              int blocks_per_cloud, void *stream) {
    if (B < 0 || N < 0 || npoint < 1)
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "fps: need B >= 0, N >= 0, npoint >= 1 (got %lld, %lld, %lld)",
                    (long long)B, (long long)N, (long long)npoint);
    if (strategy < PC_FPS_AUTO || strategy > PC_FPS_GRID)
        return fail(PC_ERR_INVALID_ARGUMENT, "fps: unknown strategy %d", strategy);
    if (cluster_size < 0 || cluster_size > 16 || blocks_per_cloud < 0)
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "fps: cluster_size must be 0..16 and blocks_per_cloud >= 0");
    if (B == 0) return PC_OK;
    if (N < 1 || start_idx < 0 || start_idx >= N)
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "fps: need 0 <= start_idx < N (got start_idx=%lld, N=%lld)",
                    (long long)start_idx, (long long)N);
    if (N > kMaxInt || npoint > kMaxInt || B > kMaxInt || !mul_ok(B, N, 3) ||
        !mul_ok(B, npoint, 1))
        return fail(PC_ERR_UNSUPPORTED, "fps: sizes beyond 32-bit indexing");
    const pcn::DeviceInfo *dev = nullptr;
    int rc = current_device(&dev);
    if (rc != PC_OK) return rc;
    if ((rc = check_ptr(xyz, dev->device, 4, "xyz")) != PC_OK) return rc;
    if ((rc = check_ptr(out_idx, dev->device, 8, "out_idx")) != PC_OK) return rc;
    pcn::FpsPlan plan =
        pcn::plan_fps(*dev, B, N, strategy, cluster_size, blocks_per_cloud);
    if (!plan.ok)
        return fail(PC_ERR_UNSUPPORTED, "fps: %s (B=%lld, N=%lld)", plan.why,
                    (long long)B, (long long)N);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *ws = workspace;
    bool owned = false;
    if (plan.workspace_bytes > 0) {
        if (ws != nullptr) {
            if (workspace_bytes < plan.workspace_bytes)
                return fail(PC_ERR_INVALID_ARGUMENT,
                            "fps: workspace of %zu bytes, need %zu",
                            workspace_bytes, plan.workspace_bytes);
            if ((rc = check_ptr(ws, dev->device, 256, "workspace")) != PC_OK)
                return rc;
        } else {
            cudaError_t e = pcn::scratch_alloc(*dev, &ws, plan.workspace_bytes, st);
            if (e != cudaSuccess) return cuda_fail(e, "fps: workspace allocation");
            owned = true;
        }
    }
    cudaError_t e = pcn::launch_fps(*dev, plan, xyz, B, N, npoint, start_idx,
                                    out_idx, ws, st);
    if (owned) {
        cudaError_t e2 = pcn::scratch_free(ws, st);
        if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e, "fps: launch");
    return PC_OK;
}

int pc_fps(const float *xyz, int64_t B, int64_t N, int64_t npoint,
           int64_t start_idx, int64_t *out_idx, void *workspace,
           size_t workspace_bytes, void *stream) {
    return pc_fps_ex(xyz, B, N, npoint, start_idx, out_idx, workspace,
                     workspace_bytes, PC_FPS_AUTO, 0, 0, stream);
}

// Shared validation and launch of kNN; `strict` enforces the plain
// operator's k <= N rule (the ex form pads instead).
static int knn_common(const char *name, const float *query, int64_t B,
                      int64_t Q, const float *ref, int64_t N, int64_t k,
                      const int64_t *q_len, const int64_t *r_len, int flags,
                      bool strict, float *out_dist, int64_t *out_idx,
                      void *stream) {
    if (B < 0 || Q < 0 || N < 0)
        return fail(PC_ERR_INVALID_ARGUMENT, "%s: negative size", name);
    if (k < 1 || (strict && k > N))
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "%s: need 1 <= k <= N (got k=%lld, N=%lld)", name,
                    (long long)k, (long long)N);
    if ((flags & ~PC_KNN_SQUARED) != 0)
        return fail(PC_ERR_INVALID_ARGUMENT, "%s: unknown flags 0x%x", name, flags);
    if (k > 256)
        return fail(PC_ERR_UNSUPPORTED, "%s: k=%lld above the maximum 256", name,
                    (long long)k);
    if (B > 65535)
        return fail(PC_ERR_UNSUPPORTED, "%s: B=%lld above 65535", name, (long long)B);
    if (Q > kMaxInt || N > kMaxInt || !mul_ok(B, Q, k) || !mul_ok(B, N, 3) ||
        !mul_ok(B, Q, 3))
        return fail(PC_ERR_UNSUPPORTED, "%s: sizes beyond 32-bit indexing", name);
    if (B == 0 || Q == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    int rc = current_device(&dev);
    if (rc != PC_OK) return rc;
    if ((rc = check_ptr(query, dev->device, 4, "query")) != PC_OK) return rc;
    if (N > 0 && (rc = check_ptr(ref, dev->device, 4, "ref")) != PC_OK) return rc;
    if ((rc = check_ptr(out_dist, dev->device, 4, "out_dist")) != PC_OK) return rc;
    if ((rc = check_ptr(out_idx, dev->device, 8, "out_idx")) != PC_OK) return rc;
    if (q_len && (rc = check_ptr(q_len, dev->device, 8, "query_lengths")) != PC_OK)
        return rc;
    if (r_len && (rc = check_ptr(r_len, dev->device, 8, "ref_lengths")) != PC_OK)
        return rc;
    cudaError_t e = pcn::launch_knn(*dev, query, B, Q, ref, N, int(k), q_len,
                                    r_len, (flags & PC_KNN_SQUARED) != 0,
                                    out_dist, out_idx,
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "knn: launch");
    return PC_OK;
}

int pc_knn(const float *query, int64_t B, int64_t Q, const float *ref,
           int64_t N, int64_t k, float *out_dist, int64_t *out_idx,
           void *stream) {
    return knn_common("knn", query, B, Q, ref, N, k, nullptr, nullptr, 0, true,
                      out_dist, out_idx, stream);
}

int pc_knn_ex(const float *query, int64_t B, int64_t Q, const float *ref,
              int64_t N, int64_t k, const int64_t *query_lengths,
              const int64_t *ref_lengths, int flags, float *out_dist,
              int64_t *out_idx, void *stream) {
    return knn_common("knn_ex", query, B, Q, ref, N, k, query_lengths,
                      ref_lengths, flags, false, out_dist, out_idx, stream);
}

static int bq_common(const char *name, const float *query, int64_t B,
                     int64_t Q, const float *ref, int64_t N,
                     const int64_t *q_len, const int64_t *r_len, double radius,
                     int64_t K, float *out_dist2, int64_t *out_idx,
                     void *stream) {
    if (B < 0 || Q < 0 || N < 0)
        return fail(PC_ERR_INVALID_ARGUMENT, "%s: negative size", name);
    if (!std::isfinite(radius) || !(radius > 0.0))
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "%s: radius must be finite and > 0 (got %g)", name, radius);
    if (K < 1)
        return fail(PC_ERR_INVALID_ARGUMENT, "%s: need K >= 1 (got %lld)", name,
                    (long long)K);
    if (B > 65535)
        return fail(PC_ERR_UNSUPPORTED, "%s: B=%lld above 65535", name,
                    (long long)B);
    if (Q > kMaxInt || N > kMaxInt || K > kMaxInt || !mul_ok(B, Q, K) ||
        !mul_ok(B, N, 3) || !mul_ok(B, Q, 3))
        return fail(PC_ERR_UNSUPPORTED, "%s: sizes beyond 32-bit indexing", name);
    if (B == 0 || Q == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    int rc = current_device(&dev);
    if (rc != PC_OK) return rc;
    if ((rc = check_ptr(query, dev->device, 4, "query")) != PC_OK) return rc;
    if (N > 0 && (rc = check_ptr(ref, dev->device, 4, "ref")) != PC_OK) return rc;
    if ((rc = check_ptr(out_dist2, dev->device, 4, "out_dist2")) != PC_OK) return rc;
    if ((rc = check_ptr(out_idx, dev->device, 8, "out_idx")) != PC_OK) return rc;
    if (q_len && (rc = check_ptr(q_len, dev->device, 8, "query_lengths")) != PC_OK)
        return rc;
    if (r_len && (rc = check_ptr(r_len, dev->device, 8, "ref_lengths")) != PC_OK)
        return rc;
    const float r32 = static_cast<float>(radius);
    cudaError_t e = pcn::launch_ball_query(*dev, query, B, Q, ref, N, q_len,
                                           r_len, r32, K, out_dist2, out_idx,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "ball_query: launch");
    return PC_OK;
}

int pc_ball_query(const float *query, int64_t B, int64_t Q, const float *ref,
                  int64_t N, double radius, int64_t K, float *out_dist2,
                  int64_t *out_idx, void *stream) {
    return bq_common("ball_query", query, B, Q, ref, N, nullptr, nullptr,
                     radius, K, out_dist2, out_idx, stream);
}

int pc_ball_query_ex(const float *query, int64_t B, int64_t Q,
                     const float *ref, int64_t N, const int64_t *query_lengths,
                     const int64_t *ref_lengths, double radius, int64_t K,
                     float *out_dist2, int64_t *out_idx, void *stream) {
    return bq_common("ball_query_ex", query, B, Q, ref, N, query_lengths,
                     ref_lengths, radius, K, out_dist2, out_idx, stream);
}

// kNN and Ball Query of one query set against one reference set: the checks
// of pc_knn and pc_ball_query together.
static int knn_bq_check(const char *name, int64_t B, int64_t Q, int64_t N, int64_t k,
                        double radius, int64_t K) {
    if (B < 0 || Q < 0 || N < 0)
        return fail(PC_ERR_INVALID_ARGUMENT, "%s: negative size", name);
    if (k < 1 || k > N)
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "%s: need 1 <= k <= N (got k=%lld, N=%lld)", name, (long long)k,
                    (long long)N);
    if (!std::isfinite(radius) || !(radius > 0.0))
        return fail(PC_ERR_INVALID_ARGUMENT,
                    "%s: radius must be finite and > 0 (got %g)", name, radius);
    if (K < 1)
        return fail(PC_ERR_INVALID_ARGUMENT, "%s: need K >= 1 (got %lld)", name,
                    (long long)K);
    if (k > 256)
        return fail(PC_ERR_UNSUPPORTED, "%s: k=%lld above the maximum 256", name,
                    (long long)k);
    if (B > 65535)
        return fail(PC_ERR_UNSUPPORTED, "%s: B=%lld above 65535", name, (long long)B);
    if (Q > kMaxInt || N > kMaxInt || K > kMaxInt || !mul_ok(B, Q, k) ||
        !mul_ok(B, Q, K) || !mul_ok(B, N, 3) || !mul_ok(B, Q, 3))
        return fail(PC_ERR_UNSUPPORTED, "%s: sizes beyond 32-bit indexing", name);
    return PC_OK;
}

int pc_knn_ball_query(const float *query, int64_t B, int64_t Q, const float *ref,
                      int64_t N, int64_t k, float *knn_dist, int64_t *knn_idx,
                      double radius, int64_t K, float *bq_dist2, int64_t *bq_idx,
                      void *stream) {
    int rc = knn_bq_check("knn_ball_query", B, Q, N, k, radius, K);
    if (rc != PC_OK) return rc;
    if (B == 0 || Q == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    if ((rc = current_device(&dev)) != PC_OK) return rc;
    if ((rc = check_ptr(query, dev->device, 4, "query")) != PC_OK) return rc;
    if ((rc = check_ptr(ref, dev->device, 4, "ref")) != PC_OK) return rc;
    if ((rc = check_ptr(knn_dist, dev->device, 4, "knn_dist")) != PC_OK) return rc;
    if ((rc = check_ptr(knn_idx, dev->device, 8, "knn_idx")) != PC_OK) return rc;
    if ((rc = check_ptr(bq_dist2, dev->device, 4, "bq_dist2")) != PC_OK) return rc;
    if ((rc = check_ptr(bq_idx, dev->device, 8, "bq_idx")) != PC_OK) return rc;
    const cudaError_t e = pcn::launch_knn_ball_query(
        *dev, query, B, Q, ref, N, int(k), knn_dist, knn_idx, static_cast<float>(radius),
        K, bq_dist2, bq_idx, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "knn_ball_query: launch");
    return PC_OK;
}

int pc_knn_ball_query_plan(int64_t B, int64_t Q, int64_t N, int64_t k, double radius,
                           int64_t K, int *out_fused) {
    if (out_fused == nullptr)
        return fail(PC_ERR_INVALID_ARGUMENT, "knn_ball_query_plan: out_fused is NULL");
    *out_fused = 0;
    int rc = knn_bq_check("knn_ball_query_plan", B, Q, N, k, radius, K);
    if (rc != PC_OK) return rc;
    const pcn::DeviceInfo *dev = nullptr;
    if ((rc = current_device(&dev)) != PC_OK) return rc;
    *out_fused = B > 0 && Q > 0 &&
                 pcn::knn_ball_query_fused(*dev, B, Q, N, int(k),
                                           static_cast<float>(radius), K);
    return PC_OK;
}

int pc_device_status(void *stream, int reset, int32_t *out_status) {
    if (out_status == nullptr)
        return fail(PC_ERR_INVALID_ARGUMENT, "device_status: out_status is NULL");
    const pcn::DeviceInfo *dev = nullptr;
    int rc = current_device(&dev);
    if (rc != PC_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "device_status: synchronize");
    int v = 0;
    e = cudaMemcpy(&v, dev->status_word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "device_status: read");
    if (reset && v != 0) {
        e = cudaMemset(dev->status_word, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "device_status: reset");
    }
    *out_status = v;
    return PC_OK;
}

}  // extern "C"
