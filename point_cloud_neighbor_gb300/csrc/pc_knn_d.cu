// pc_knn_d.cu -- exact brute-force kNN in D dimensions on sm_103a.
//
// Operator (mps-pointops project page, "Roadmap", Phase 2: kNN in arbitrary
// dimension for feature-space neighbour search, with "direct
// dimension-by-dimension distance accumulation as the numerical baseline"):
//   s = fl(... fl(fl(t_0 + t_1) + t_2) ... + t_{D-1}),  t_d = fl(fl(q_d - x_d)^2),
// accumulated in increasing d with separately rounded float32 operations
// (for D = 3 this is the s32 of the point operators); the k smallest (s, j)
// in lexicographic order, D = sqrt(s) or s (PC_KNN_SQUARED).
//
// Design (one launch; k <= 32, D <= 256):
//  * A block owns KD_QT = 64 queries of one cloud and has KD_PH = 4 phases of
//    64 threads: thread (phase p, query q) examines the references whose
//    position in each tile of KD_RT = 32 falls in [8p, 8p + 8).  Query rows
//    sit in shared memory with a padded stride (128-bit loads of 32 different
//    rows by a warp are conflict-free); reference tiles are loaded by the
//    whole block and read as broadcasts (a warp's lanes share a phase).
//  * A thread accumulates 4 references at once, 4 dimensions per step, in
//    strict dimension order per pair (zero-padded dimensions add +0 and leave
//    s unchanged), and keeps a max-heap of its k best (s, j) in shared memory
//    (entry e of thread t at [e * 256 + t]).
//  * At the end the phase-0 thread of each query inserts the other phases'
//    entries into its heap (the same total order, so the result is exact),
//    heap-sorts it and writes the row.
#include "pointcloud.h"
#include "pc_device.cuh"
#include "pc_internal.h"

#include <algorithm>
#include <climits>
#include <cstdio>

namespace pcn {
namespace {

constexpr int KD_THREADS = 256;
constexpr int KD_QT = 64;
constexpr int KD_PH = KD_THREADS / KD_QT;
constexpr int KD_RT = 32;
constexpr int KD_MAXK = 32;
constexpr int KD_MAXD = 256;

// Row stride in floats: a multiple of 4 with (stride / 4) odd, so that 8
// consecutive rows read with 128-bit loads hit distinct bank groups.
__host__ __device__ constexpr int kd_stride(int D) { return ((D + 7) / 8) * 8 + 4; }

__host__ __device__ constexpr size_t kd_smem(int D, int k) {
    return size_t(KD_QT + KD_RT) * kd_stride(D) * sizeof(float) +
           size_t(KD_THREADS) * k * 8;
}

struct KnnDArgs {
    const float *query;
    const float *ref;
    int Q, N, D, k;
    int squared;
    float *out_dist;
    int64_t *out_idx;
};

__device__ __forceinline__ bool kd_after(float as, int aj, float bs, int bj) {
    return as > bs || (as == bs && aj > bj);
}

// Sift (s, j) down from the root of the max-heap hs/hj of n entries whose
// entries are `stride` apart.
__device__ __forceinline__ void kd_sift(float *hs, int *hj, int n, int stride,
                                        int pos, float s, int j) {
    for (;;) {
        int c = 2 * pos + 1;
        if (c >= n) break;
        float cs = hs[c * stride];
        int cj = hj[c * stride];
        if (c + 1 < n) {
            const float ds = hs[(c + 1) * stride];
            const int dj = hj[(c + 1) * stride];
            if (kd_after(ds, dj, cs, cj)) {
                ++c;
                cs = ds;
                cj = dj;
            }
        }
        if (!kd_after(cs, cj, s, j)) break;
        hs[pos * stride] = cs;
        hj[pos * stride] = cj;
        pos = c;
    }
    hs[pos * stride] = s;
    hj[pos * stride] = j;
}

__global__ void __launch_bounds__(KD_THREADS) knn_d_kernel(const KnnDArgs a) {
    extern __shared__ __align__(16) float kd_smem_f[];
    const int D = a.D, k = a.k;
    const int S = kd_stride(D);
    const int D4 = (D + 3) / 4;
    float *qt = kd_smem_f;                      // [KD_QT][S]
    float *rt = qt + KD_QT * S;                 // [KD_RT][S]
    float *hs_all = rt + KD_RT * S;             // [k][KD_THREADS]
    int *hj_all = reinterpret_cast<int *>(hs_all + size_t(k) * KD_THREADS);
    const int b = blockIdx.y;
    const int q0 = blockIdx.x * KD_QT;
    const int tid = threadIdx.x;
    const int ql = tid % KD_QT, phase = tid / KD_QT;
    const float inf = __int_as_float(0x7f800000);

    // query rows (zero padded)
    const float *qg = a.query + (size_t(b) * a.Q + q0) * D;
    const int nq = min(KD_QT, a.Q - q0);
    for (int e = tid; e < KD_QT * S; e += KD_THREADS) {
        const int r = e / S, d = e % S;
        qt[e] = (r < nq && d < D) ? qg[size_t(r) * D + d] : 0.0f;
    }
    float *hs = hs_all + tid;
    int *hj = hj_all + tid;
    for (int e = 0; e < k; ++e) {
        hs[e * KD_THREADS] = inf;
        hj[e * KD_THREADS] = INT_MAX;
    }
    float ts = inf;
    int tj = INT_MAX;

    const float *xg = a.ref + size_t(b) * a.N * D;
    const float4 *qrow = reinterpret_cast<const float4 *>(qt + ql * S);
    for (int j0 = 0; j0 < a.N; j0 += KD_RT) {
        __syncthreads();  // the previous tile is no longer read
        const int nr = min(KD_RT, a.N - j0);
        for (int e = tid; e < KD_RT * S; e += KD_THREADS) {
            const int r = e / S, d = e % S;
            rt[e] = (r < nr && d < D) ? xg[size_t(j0 + r) * D + d] : 0.0f;
        }
        __syncthreads();
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
            const int r0 = phase * 8 + g * 4;  // 4 references of this thread
            if (r0 >= nr) break;
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            const float4 *x0 = reinterpret_cast<const float4 *>(rt + r0 * S);
            for (int d4 = 0; d4 < D4; ++d4) {
                const float4 qv = qrow[d4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 xv = x0[u * (S / 4) + d4];
                    float t = __fsub_rn(qv.x, xv.x);
                    s[u] = __fadd_rn(s[u], __fmul_rn(t, t));
                    t = __fsub_rn(qv.y, xv.y);
                    s[u] = __fadd_rn(s[u], __fmul_rn(t, t));
                    t = __fsub_rn(qv.z, xv.z);
                    s[u] = __fadd_rn(s[u], __fmul_rn(t, t));
                    t = __fsub_rn(qv.w, xv.w);
                    s[u] = __fadd_rn(s[u], __fmul_rn(t, t));
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + r0 + u;
                if (r0 + u < nr && kd_after(ts, tj, s[u], j)) {
                    kd_sift(hs, hj, k, KD_THREADS, 0, s[u], j);
                    ts = hs[0];
                    tj = hj[0];
                }
            }
        }
    }
    __syncthreads();
    if (phase != 0 || ql >= nq) return;
    // merge the other phases' heaps of this query into this one
    for (int p = 1; p < KD_PH; ++p) {
        const int other = p * KD_QT + ql;
        for (int e = 0; e < k; ++e) {
            const float sv = hs_all[e * KD_THREADS + other];
            const int jv = hj_all[e * KD_THREADS + other];
            if (kd_after(ts, tj, sv, jv)) {
                kd_sift(hs, hj, k, KD_THREADS, 0, sv, jv);
                ts = hs[0];
                tj = hj[0];
            }
        }
    }
    for (int n = k - 1; n > 0; --n) {  // heap sort into ascending order
        const float sv = hs[n * KD_THREADS];
        const int jv = hj[n * KD_THREADS];
        hs[n * KD_THREADS] = hs[0];
        hj[n * KD_THREADS] = hj[0];
        kd_sift(hs, hj, n, KD_THREADS, 0, sv, jv);
    }
    const size_t row = size_t(b) * a.Q + q0 + ql;
    for (int e = 0; e < k; ++e) {
        const float sv = hs[e * KD_THREADS];
        a.out_idx[row * k + e] = hj[e * KD_THREADS];
        a.out_dist[row * k + e] = a.squared ? sv : __fsqrt_rn(sv);
    }
}

}  // namespace
}  // namespace pcn

extern "C" int pc_knn_d(const float *query, int64_t B, int64_t Q,
                        const float *ref, int64_t N, int64_t D, int64_t k,
                        int flags, float *out_dist, int64_t *out_idx,
                        void *stream) {
    char m[200];
    if (B < 0 || Q < 0 || N < 0 || D < 1)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, "knn_d: negative size or D < 1");
    if (k < 1 || k > N) {
        std::snprintf(m, sizeof(m), "knn_d: need 1 <= k <= N (got k=%lld, N=%lld)",
                      (long long)k, (long long)N);
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, m);
    }
    if ((flags & ~PC_KNN_SQUARED) != 0)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, "knn_d: unknown flags");
    if (k > pcn::KD_MAXK || D > pcn::KD_MAXD || B > 65535 || Q > 2147483647 ||
        N > 2147483647 || B * std::max(Q, N) * D > (int64_t(1) << 40)) {
        std::snprintf(m, sizeof(m),
                      "knn_d: supported k <= %d, D <= %d, 32-bit indexing (got k=%lld, D=%lld)",
                      pcn::KD_MAXK, pcn::KD_MAXD, (long long)k, (long long)D);
        return pcn::api_fail(PC_ERR_UNSUPPORTED, m);
    }
    if (B == 0 || Q == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    int rc = pcn::api_current_device(&dev);
    if (rc != PC_OK) return rc;
    const int d = dev->device;
    if ((rc = pcn::api_check_ptr(query, d, 4, "query")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(ref, d, 4, "ref")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(out_dist, d, 4, "out_dist")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(out_idx, d, 8, "out_idx")) != PC_OK) return rc;
    pcn::KnnDArgs a{};
    a.query = query;
    a.ref = ref;
    a.Q = int(Q);
    a.N = int(N);
    a.D = int(D);
    a.k = int(k);
    a.squared = (flags & PC_KNN_SQUARED) != 0;
    a.out_dist = out_dist;
    a.out_idx = out_idx;
    const size_t smem = pcn::kd_smem(int(D), int(k));
    cudaError_t e = cudaFuncSetAttribute(pcn::knn_d_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e == cudaSuccess) {
        const dim3 grid(unsigned((Q + pcn::KD_QT - 1) / pcn::KD_QT), unsigned(B));
        pcn::knn_d_kernel<<<grid, pcn::KD_THREADS, smem,
                            static_cast<cudaStream_t>(stream)>>>(a);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        std::snprintf(m, sizeof(m), "knn_d: %s", cudaGetErrorString(e));
        return pcn::api_fail(PC_ERR_CUDA, m);
    }
    return PC_OK;
}
