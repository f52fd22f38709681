// pc_chamfer.cu -- bidirectional squared-L2 Chamfer distance (forward) on
// sm_103a.
//
// The mps-pointops project page ("Quick start"; "Roadmap", Phase 4) defines
// L = sum_i |q_i - x_a(i)|^2 + sum_j |x_j - q_b(j)|^2 with a(i) the nearest
// point of the second cloud to q_i and b(j) the nearest point of the first
// cloud to x_j, lengths masks for padding, per-cloud weights and point and
// batch reductions.  Here:
//   * each direction is the brute-force kNN kernel (pc_knn.cu) with k = 1,
//     the clouds' valid lengths and the squared distance returned: nearest
//     index and s32 with exact ties to the smaller index; the two directions
//     share one launch;
//   * one block of 1024 threads per cloud reduces its per-point distances in
//     float64 in a fixed order (four strided partial sums per thread, then a
//     fixed shuffle tree), and one more block sums the clouds' losses in the
//     same way, so the loss is deterministic from run to run and within a few
//     float64 roundings of the exact sum before its single rounding to
//     float32.
// Readings: a point with no valid reference contributes 0 (index -1);
// "mean" over points divides a cloud's sum by max(length, 1); weights scale
// each cloud's loss; "mean" over the batch divides by B (0 for B = 0).
#include "pointcloud.h"
#include "pc_internal.h"

#include <cstdio>

namespace pcn {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int RED_THREADS = 1024;

struct ChamferReduceArgs {
    const float *dist_x;     // [B, P1]
    const float *dist_y;     // [B, P2], NULL when single-directional
    const int64_t *x_len, *y_len;
    const float *weights;    // [B] or NULL
    int B, P1, P2;
    int point_mean;          // 1: mean over points, 0: sum
    int batch_mode;          // PC_REDUCTION_NONE / SUM / MEAN
    float *out_loss;
    double *cloud_loss;      // [B] scratch (SUM / MEAN)
};

__device__ __forceinline__ int valid_len(const int64_t *lens, int b, int full) {
    if (lens == nullptr) return full;
    const int64_t v = lens[b];
    return v < 0 ? 0 : (v > full ? full : static_cast<int>(v));
}

// Sum of v[0..n) in float64 over the whole block, in a fixed order (four
// strided partial sums per thread, so that four loads are in flight); the
// result is returned to every thread.
template <class T>
__device__ double block_sum(const T *v, int n, double *part) {
    double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
    int i = threadIdx.x;
    for (; i + 3 * RED_THREADS < n; i += 4 * RED_THREADS) {
        a0 += double(v[i]);
        a1 += double(v[i + RED_THREADS]);
        a2 += double(v[i + 2 * RED_THREADS]);
        a3 += double(v[i + 3 * RED_THREADS]);
    }
    for (; i < n; i += RED_THREADS) a0 += double(v[i]);
    double acc = (a0 + a1) + (a2 + a3);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(FULL, acc, o);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) part[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        double w = part[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w += __shfl_down_sync(FULL, w, o);
        if (lane == 0) part[32] = w;
    }
    __syncthreads();
    const double r = part[32];
    __syncthreads();
    return r;
}

// One block per cloud: its loss, into out_loss[b] (NONE) or cloud_loss[b].
__global__ void __launch_bounds__(RED_THREADS)
chamfer_reduce_kernel(const ChamferReduceArgs a) {
    __shared__ double part[33];
    const int b = blockIdx.x;
    const int nx = valid_len(a.x_len, b, a.P1);
    double t = block_sum(a.dist_x + size_t(b) * a.P1, nx, part);
    if (a.point_mean) t = t / double(max(nx, 1));
    if (a.dist_y != nullptr) {
        const int ny = valid_len(a.y_len, b, a.P2);
        double u = block_sum(a.dist_y + size_t(b) * a.P2, ny, part);
        if (a.point_mean) u = u / double(max(ny, 1));
        t = t + u;
    }
    if (a.weights != nullptr) t = t * double(a.weights[b]);
    if (threadIdx.x == 0) {
        if (a.batch_mode == PC_REDUCTION_NONE)
            a.out_loss[b] = float(t);
        else
            a.cloud_loss[b] = t;
    }
}

// The batch reduction (SUM / MEAN) over the clouds' losses, one block.
__global__ void __launch_bounds__(RED_THREADS)
chamfer_batch_kernel(const ChamferReduceArgs a) {
    __shared__ double part[33];
    const double total = block_sum(a.cloud_loss, a.B, part);
    if (threadIdx.x == 0)
        a.out_loss[0] = a.batch_mode == PC_REDUCTION_SUM
                            ? float(total)
                            : (a.B > 0 ? float(total / double(a.B)) : 0.0f);
}

}  // namespace
}  // namespace pcn

namespace {

int fail_msg(int code, const char *fmt, long long v) {
    char m[200];
    std::snprintf(m, sizeof(m), fmt, v);
    return pcn::api_fail(code, m);
}

}  // namespace

extern "C" int pc_chamfer(const float *x, int64_t B, int64_t P1,
                          const float *y, int64_t P2, const int64_t *x_lengths,
                          const int64_t *y_lengths, const float *weights,
                          int point_reduction, int batch_reduction,
                          int single_directional, float *out_dist_x,
                          int64_t *out_idx_x, float *out_dist_y,
                          int64_t *out_idx_y, float *out_loss, void *stream) {
    constexpr int64_t kMaxInt = 2147483647;
    if (B < 0 || P1 < 0 || P2 < 0)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, "chamfer: negative size");
    if (B > 65535) return fail_msg(PC_ERR_UNSUPPORTED, "chamfer: B=%lld above 65535", B);
    if (P1 > kMaxInt || P2 > kMaxInt || B * (P1 > P2 ? P1 : P2) > (int64_t(1) << 40))
        return pcn::api_fail(PC_ERR_UNSUPPORTED, "chamfer: sizes beyond 32-bit indexing");
    if (out_loss != nullptr) {
        if (point_reduction != PC_REDUCTION_SUM && point_reduction != PC_REDUCTION_MEAN)
            return fail_msg(PC_ERR_INVALID_ARGUMENT,
                            "chamfer: point_reduction must be SUM or MEAN (got %lld)",
                            point_reduction);
        if (batch_reduction != PC_REDUCTION_NONE && batch_reduction != PC_REDUCTION_SUM &&
            batch_reduction != PC_REDUCTION_MEAN)
            return fail_msg(PC_ERR_INVALID_ARGUMENT,
                            "chamfer: batch_reduction must be NONE, SUM or MEAN (got %lld)",
                            batch_reduction);
    }
    const bool both = single_directional == 0;
    if (B == 0 && (out_loss == nullptr || batch_reduction == PC_REDUCTION_NONE))
        return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    int rc = pcn::api_current_device(&dev);
    if (rc != PC_OK) return rc;
    const int d = dev->device;
    if (B > 0 && P1 > 0) {
        if ((rc = pcn::api_check_ptr(x, d, 4, "x")) != PC_OK) return rc;
        if ((rc = pcn::api_check_ptr(out_dist_x, d, 4, "out_dist_x")) != PC_OK) return rc;
        if ((rc = pcn::api_check_ptr(out_idx_x, d, 8, "out_idx_x")) != PC_OK) return rc;
    }
    if (B > 0 && P2 > 0) {
        if ((rc = pcn::api_check_ptr(y, d, 4, "y")) != PC_OK) return rc;
        if (both) {
            if ((rc = pcn::api_check_ptr(out_dist_y, d, 4, "out_dist_y")) != PC_OK) return rc;
            if ((rc = pcn::api_check_ptr(out_idx_y, d, 8, "out_idx_y")) != PC_OK) return rc;
        }
    }
    if (x_lengths && (rc = pcn::api_check_ptr(x_lengths, d, 8, "x_lengths")) != PC_OK)
        return rc;
    if (y_lengths && (rc = pcn::api_check_ptr(y_lengths, d, 8, "y_lengths")) != PC_OK)
        return rc;
    if (weights && (rc = pcn::api_check_ptr(weights, d, 4, "weights")) != PC_OK) return rc;
    if (out_loss && (rc = pcn::api_check_ptr(out_loss, d, 4, "out_loss")) != PC_OK)
        return rc;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (both && B > 0 && P1 > 0 && P2 > 0) {
        // both directions in one launch: twice the blocks of either alone
        e = pcn::launch_knn_pair(*dev, B, 1, true, x, P1, y, P2, x_lengths,
                                 y_lengths, out_dist_x, out_idx_x, y, P2, x, P1,
                                 y_lengths, x_lengths, out_dist_y, out_idx_y, st);
    } else {
        if (B > 0 && P1 > 0)
            e = pcn::launch_knn(*dev, x, B, P1, y, P2, 1, x_lengths, y_lengths, true,
                                out_dist_x, out_idx_x, st);
        if (e == cudaSuccess && both && B > 0 && P2 > 0)
            e = pcn::launch_knn(*dev, y, B, P2, x, P1, 1, y_lengths, x_lengths, true,
                                out_dist_y, out_idx_y, st);
    }
    if (e == cudaSuccess && out_loss != nullptr) {
        pcn::ChamferReduceArgs a{};
        a.dist_x = P1 > 0 ? out_dist_x : nullptr;
        a.dist_y = both ? (P2 > 0 ? out_dist_y : nullptr) : nullptr;
        a.x_len = x_lengths;
        a.y_len = y_lengths;
        a.weights = weights;
        a.B = int(B);
        a.P1 = int(P1);
        a.P2 = int(P2);
        a.point_mean = point_reduction == PC_REDUCTION_MEAN;
        a.batch_mode = batch_reduction;
        a.out_loss = out_loss;
        if (batch_reduction == PC_REDUCTION_NONE) {
            if (B > 0) pcn::chamfer_reduce_kernel<<<unsigned(B), pcn::RED_THREADS, 0, st>>>(a);
            e = cudaGetLastError();
        } else {
            // the clouds' losses in stream-ordered scratch, then their sum
            double *cl = nullptr;
            e = pcn::scratch_alloc(*dev, reinterpret_cast<void **>(&cl),
                                   size_t(B > 0 ? B : 1) * sizeof(double), st);
            if (e == cudaSuccess) {
                a.cloud_loss = cl;
                if (B > 0)
                    pcn::chamfer_reduce_kernel<<<unsigned(B), pcn::RED_THREADS, 0, st>>>(a);
                pcn::chamfer_batch_kernel<<<1, pcn::RED_THREADS, 0, st>>>(a);
                e = cudaGetLastError();
                const cudaError_t f = pcn::scratch_free(cl, st);
                if (e == cudaSuccess) e = f;
            }
        }
    }
    if (e != cudaSuccess) {
        char m[200];
        std::snprintf(m, sizeof(m), "chamfer: %s", cudaGetErrorString(e));
        return pcn::api_fail(PC_ERR_CUDA, m);
    }
    return PC_OK;
}
