// pc_fps_static.cu -- farthest point sampling for callers that cannot
// allocate device memory.
//
// pc_fps's grid schedule exchanges one 64-bit word per block and step through
// scratch memory, which pc_fps takes from the caller or allocates itself.
// Some callers can do neither at call time: a host application that has
// handed (nearly) all device memory to its own pool, so that cudaMalloc /
// cudaMallocAsync would fail or break its accounting, or a real-time loop
// with a fixed memory footprint that forbids allocation after start-up.
// pc_fps_grid_static serves them: its scratch is a file-scope __device__
// array that exists, at a fixed size, on every device that loads this library
// until the process exits.  The call itself allocates nothing.
//
// Host code must not hand g_fps_static_scratch to a kernel by name: on the
// host that name is only a stand-in for the device array.  Its device
// address is looked up once per device with cudaGetSymbolAddress (on the
// first call made while that device is current) and cached.
#include "pointcloud.h"
#include "pc_internal.h"

#include <cstdio>
#include <mutex>

namespace {

// 16384 exchange words (128 KiB) per device.  The step-by-step grid
// schedule uses B * max(2 * blocks per cloud, 32 * clusters per cloud)
// words, and the blocks never exceed the SM count, so this covers any device
// with up to 8192 SMs; the rounds take B * 2 * clusters * 4128 bytes (one
// cloud in up to 15 clusters) and fall back to the step-by-step kernel
// beyond that.
constexpr size_t kStaticScratchWords = 16384;
static __device__ __align__(256) uint64_t g_fps_static_scratch[kStaticScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
void *g_static_addr[kMaxDevices] = {};

// Device address of this device's scratch array (resolved once per device
// and kept until the process exits: a cudaDeviceReset, which unloads the
// library's device code, leaves the cached address stale).
int static_scratch_address(int device, void **out) {
    if (device < 0 || device >= kMaxDevices) {
        char msg[128];
        std::snprintf(msg, sizeof(msg),
                      "fps_grid_static: device ordinal %d beyond the %d this "
                      "entry point serves", device, kMaxDevices);
        return pcn::api_fail(PC_ERR_UNSUPPORTED, msg);
    }
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (g_static_addr[device] == nullptr) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_fps_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            char msg[256];
            std::snprintf(msg, sizeof(msg),
                          "fps_grid_static: cudaGetSymbolAddress failed: %s",
                          cudaGetErrorString(e));
            return pcn::api_fail(PC_ERR_CUDA, msg);
        }
        g_static_addr[device] = p;
    }
    *out = g_static_addr[device];
    return PC_OK;
}

}  // namespace

extern "C" int pc_fps_grid_static(const float *xyz, int64_t B, int64_t N,
                                  int64_t npoint, int64_t start_idx,
                                  int64_t *out_idx, int blocks_per_cloud,
                                  void *stream) {
    char msg[256];
    if (B < 0 || N < 0 || npoint < 1 || blocks_per_cloud < 0)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT,
                             "fps_grid_static: need B >= 0, N >= 0, npoint >= 1, "
                             "blocks_per_cloud >= 0");
    if (B == 0) return PC_OK;
    if (N < 1 || start_idx < 0 || start_idx >= N)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT,
                             "fps_grid_static: need 0 <= start_idx < N");
    if (N > 2147483647 || npoint > 2147483647 || B > 2147483647)
        return pcn::api_fail(PC_ERR_UNSUPPORTED,
                             "fps_grid_static: sizes beyond 32-bit indexing");
    const pcn::DeviceInfo *dev = nullptr;
    int rc = pcn::api_current_device(&dev);
    if (rc != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(xyz, dev->device, 4, "xyz")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(out_idx, dev->device, 8, "out_idx")) != PC_OK)
        return rc;
    pcn::FpsPlan plan =
        pcn::plan_fps(*dev, B, N, PC_FPS_GRID, 0, blocks_per_cloud);
    if (!plan.ok) {
        std::snprintf(msg, sizeof(msg), "fps_grid_static: %s", plan.why);
        return pcn::api_fail(PC_ERR_UNSUPPORTED, msg);
    }
    // the rounds kernel's summaries where they fit, else the step-by-step
    // kernel's slots
    if (plan.grid_rounds && plan.workspace_bytes > sizeof(uint64_t) * kStaticScratchWords) {
        plan.grid_rounds = false;
        plan.workspace_bytes = plan.step_workspace_bytes;
    }
    if (plan.workspace_bytes > sizeof(uint64_t) * kStaticScratchWords) {
        std::snprintf(msg, sizeof(msg),
                      "fps_grid_static: needs %zu bytes of scratch but the static "
                      "array holds %zu (%zu words: B * max(2 * blocks per cloud, "
                      "32 * clusters per cloud))",
                      plan.workspace_bytes,
                      sizeof(uint64_t) * kStaticScratchWords, kStaticScratchWords);
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, msg);
    }
    void *scratch = nullptr;
    if ((rc = static_scratch_address(dev->device, &scratch)) != PC_OK) return rc;
    // launch_fps clears the words this launch uses (cudaMemsetAsync on the same
    // stream) before the kernel, so leftovers of an earlier call do no harm.
    cudaError_t e = pcn::launch_fps(*dev, plan, xyz, B, N, npoint, start_idx,
                                    out_idx, scratch,
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        std::snprintf(msg, sizeof(msg), "fps_grid_static: launch: %s",
                      cudaGetErrorString(e));
        return pcn::api_fail(PC_ERR_CUDA, msg);
    }
    return PC_OK;
}
