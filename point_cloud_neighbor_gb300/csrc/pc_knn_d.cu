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
// Two kernels, one launch: D <= 64 knn_d_packed_kernel (below: the query
// row in registers, two references per packed instruction), else this one.
//
// knn_d_kernel (k <= 32, D <= 256):
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
    float negzero;  // -0.0f, supplied at run time (see sq2_rn)
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


// ---------------------------------------------------------------------------
// knn_d_packed_kernel<DM> (D <= DM = 64): the same arithmetic, two references
// per packed f32x2 instruction.  The thread's query row lives in registers,
// negated (x + (-q) is -(q - x) under round-to-nearest-even and the square
// removes the sign); the tile is stored dimension-major, so the thread's 8
// references of a dimension are two 128-bit broadcasts; per dimension and
// pair of references one packed add, one packed square (fma with a -0
// addend supplied at run time, see sq2_rn) and one packed accumulation, in
// increasing d -- each half the exact kernel's s bit for bit.  (The packed exact kernel with query rows in
// shared memory was bound by their per-lane loads.)
constexpr int KP_DM = 64;
constexpr int KP_STRIDE = KD_RT + 4;  // floats between dimensions of the tile

__host__ __device__ constexpr size_t kp_smem(int k) {
    return size_t(KP_DM) * KP_STRIDE * sizeof(float) + size_t(KD_THREADS) * k * 8;
}

template <int DM>
__global__ void __launch_bounds__(KD_THREADS) knn_d_packed_kernel(const KnnDArgs a) {
    extern __shared__ __align__(16) float kp_smem_f[];
    const int D = a.D, k = a.k;
    float *xt = kp_smem_f;                   // [DM][KP_STRIDE]
    float *hs_all = xt + DM * KP_STRIDE;     // [k][KD_THREADS]
    int *hj_all = reinterpret_cast<int *>(hs_all + size_t(k) * KD_THREADS);
    const int b = blockIdx.y;
    const int q0 = blockIdx.x * KD_QT;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int ql = tid % KD_QT, phase = tid / KD_QT;
    const float inf = __int_as_float(0x7f800000);
    const float2 nz = make_float2(a.negzero, a.negzero);

    const int nq = min(KD_QT, a.Q - q0);
    const bool qvalid = ql < nq;
    const float *qg = a.query + (size_t(b) * a.Q + q0 + (qvalid ? ql : 0)) * D;
    float nqr[DM];
#pragma unroll
    for (int d = 0; d < DM; ++d) nqr[d] = (qvalid && d < D) ? -qg[d] : 0.0f;
    float *hs = hs_all + tid;
    int *hj = hj_all + tid;
    for (int e = 0; e < k; ++e) {
        hs[e * KD_THREADS] = inf;
        hj[e * KD_THREADS] = INT_MAX;
    }
    float ts = inf;
    int tj = INT_MAX;
    const float *xg = a.ref + size_t(b) * a.N * D;
    const int r0 = phase * 8;  // the thread's 8 references of each tile

    for (int j0 = 0; j0 < a.N; j0 += KD_RT) {
        __syncthreads();  // the previous tile is no longer read
        const int nr = min(KD_RT, a.N - j0);
        // reference r, dimension d at xt[d * KP_STRIDE + r] (a warp per row)
        for (int r = warp; r < KD_RT; r += KD_THREADS / 32)
            for (int d = lane; d < D; d += 32)
                xt[d * KP_STRIDE + r] = r < nr ? xg[size_t(j0 + r) * D + d] : 0.0f;
        __syncthreads();
        float2 s0 = make_float2(0.f, 0.f), s1 = s0, s2 = s0, s3 = s0;
#pragma unroll
        for (int d = 0; d < DM; ++d) {
            if (d >= D) break;
            const float4 xa = *reinterpret_cast<const float4 *>(xt + d * KP_STRIDE + r0);
            const float4 xb = *reinterpret_cast<const float4 *>(xt + d * KP_STRIDE + r0 + 4);
            const float2 nqd = make_float2(nqr[d], nqr[d]);
            float2 t = __fadd2_rn(make_float2(xa.x, xa.y), nqd);
            s0 = __fadd2_rn(s0, __ffma2_rn(t, t, nz));
            t = __fadd2_rn(make_float2(xa.z, xa.w), nqd);
            s1 = __fadd2_rn(s1, __ffma2_rn(t, t, nz));
            t = __fadd2_rn(make_float2(xb.x, xb.y), nqd);
            s2 = __fadd2_rn(s2, __ffma2_rn(t, t, nz));
            t = __fadd2_rn(make_float2(xb.z, xb.w), nqd);
            s3 = __fadd2_rn(s3, __ffma2_rn(t, t, nz));
        }
        const float sv[8] = {s0.x, s0.y, s1.x, s1.y, s2.x, s2.y, s3.x, s3.y};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + r0 + u;
            if (r0 + u < nr && kd_after(ts, tj, sv[u], j)) {
                kd_sift(hs, hj, k, KD_THREADS, 0, sv[u], j);
                ts = hs[0];
                tj = hj[0];
            }
        }
    }
    __syncthreads();
    if (phase != 0 || !qvalid) return;
    // merge the other phases' heaps of this query into this one
    for (int p = 1; p < KD_PH; ++p) {
        const int other = p * KD_QT + ql;
        for (int e = 0; e < k; ++e) {
            const float sx = hs_all[e * KD_THREADS + other];
            const int jx = hj_all[e * KD_THREADS + other];
            if (kd_after(ts, tj, sx, jx)) {
                kd_sift(hs, hj, k, KD_THREADS, 0, sx, jx);
                ts = hs[0];
                tj = hj[0];
            }
        }
    }
    for (int n = k - 1; n > 0; --n) {  // heap sort into ascending order
        const float sx = hs[n * KD_THREADS];
        const int jx = hj[n * KD_THREADS];
        hs[n * KD_THREADS] = hs[0];
        hj[n * KD_THREADS] = hj[0];
        kd_sift(hs, hj, n, KD_THREADS, 0, sx, jx);
    }
    const size_t row = size_t(b) * a.Q + q0 + ql;
    for (int e = 0; e < k; ++e) {
        const float sx = hs[e * KD_THREADS];
        a.out_idx[row * k + e] = hj[e * KD_THREADS];
        a.out_dist[row * k + e] = a.squared ? sx : __fsqrt_rn(sx);
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
    a.negzero = -0.0f;
    // D <= 64: the packed kernel with the query row in registers
    const bool packed = D <= pcn::KP_DM;
    const size_t smem = packed ? pcn::kp_smem(int(k)) : pcn::kd_smem(int(D), int(k));
    const void *fn = packed
                         ? reinterpret_cast<const void *>(&pcn::knn_d_packed_kernel<pcn::KP_DM>)
                         : reinterpret_cast<const void *>(&pcn::knn_d_kernel);
    cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) {
        const dim3 grid(unsigned((Q + pcn::KD_QT - 1) / pcn::KD_QT), unsigned(B));
        if (packed)
            pcn::knn_d_packed_kernel<pcn::KP_DM><<<grid, pcn::KD_THREADS, smem,
                                                  static_cast<cudaStream_t>(stream)>>>(a);
        else
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
