// pc_ball_query.cu -- dense first-K Ball Query on sm_103a.
//
// Operator (mps-pointops project page, "Ball Query: first K within a
// radius"; "Numerical contracts", "Selection and output"): with
// R2 = fl32(fl32(r) * fl32(r)), reference j is accepted iff s < R2; the
// first K accepted indices in input order are returned with their squared
// distances, unused slots hold (-1, 0).
//
// Design (one launch, no scratch memory):
//  * A block of BQ_WARPS warps owns BQ_WARPS * G queries of one cloud; a warp
//    owns G of them, kept in shared memory as float4 (x, y, z, hits so far).
//  * Reference tiles of BQ_T = 32 * BQ_R points are staged into shared memory
//    by TMA bulk copies (double buffered) strictly in input order, then held
//    in registers: lane l holds tile points l + 32 r, so for each r the warp
//    holds 32 consecutive references in lane order.
//  * Per (query, tile) each lane evaluates BQ_R distances with packed f32x2
//    instructions and one warp vote asks whether any is inside the radius.
//    Only then, per r, a ballot gives the hits of those 32 consecutive
//    references and __popc(ballot & lanemask_lt) gives each hit its rank, so
//    a hit is written straight to slot (hits so far + rank) -- input order is
//    kept without any sort.  A query stops at K hits; the block stops reading
//    tiles when all of its queries are full.
#include "pc_device.cuh"
#include "pc_internal.h"
#include "pc_tiles.cuh"

#include <algorithm>

namespace pcn {
namespace {

constexpr int BQ_R = 8;
constexpr int BQ_T = 32 * BQ_R;
constexpr int BQ_WARPS = 8;
constexpr int BQ_THREADS = 32 * BQ_WARPS;
constexpr unsigned FULL = 0xffffffffu;

struct BqArgs {
    const float *query;
    const float *ref;
    int Q, N;
    float R2;
    int K;
    int q_per_warp;
    int ntiles;
    float *out_dist2;
    int64_t *out_idx;
    int *status;
    uint64_t timeout_ns;
    float negzero;  // -0.0f, see sq2_rn
};

__host__ __device__ constexpr size_t bq_fixed_smem() {
    return 2 * size_t(tile_buffer_bytes(BQ_T)) + 32;
}

__global__ void __launch_bounds__(BQ_THREADS, 2) bq_kernel(const BqArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const float2 nz0 = make_float2(a.negzero, a.negzero);
    const int G = a.q_per_warp;
    const int q_warp0 = (blockIdx.x * BQ_WARPS + warp) * G;
    const int nq = max(0, min(G, a.Q - q_warp0));
    const int K = a.K;

    constexpr unsigned BUF = tile_buffer_bytes(BQ_T);
    // tile buffer of stage st: smem + st * BUF
    auto tbuf = [&](int st) { return reinterpret_cast<float *>(smem + st * BUF); };
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * BUF);
    int *s_err = reinterpret_cast<int *>(smem + 2 * BUF + 16);
    float4 *qst = reinterpret_cast<float4 *>(smem + bq_fixed_smem()) + warp * G;

    const float *cref = a.ref + size_t(b) * size_t(a.N) * 3;
    const float *cq = a.query + size_t(b) * size_t(a.Q) * 3;

    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *s_err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int g = lane; g < G; g += 32) {
        float4 v = make_float4(0.f, 0.f, 0.f, __int_as_float(0));
        if (g < nq) {
            const float *p = cq + size_t(q_warp0 + g) * 3;
            v.x = p[0];
            v.y = p[1];
            v.z = p[2];
        }
        qst[g] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int it = 0; it < 2 && it < a.ntiles; ++it) {
            const int j0 = it * BQ_T;
            issue_tile(tbuf(it), cref + size_t(j0) * 3, min(BQ_T, a.N - j0),
                       &bars[it]);
        }
    }

    int ndone = 0;  // queries of this warp holding K hits
    int failed_it = -1, stop_it = a.ntiles;
    for (int it = 0; it < a.ntiles; ++it) {
        const int st = it & 1;
        const unsigned par = (it >> 1) & 1;
        if (!mbar_wait_bounded(&bars[st], par, a.timeout_ns)) *s_err = 1;
        const int j0 = it * BQ_T;
        const int cnt = min(BQ_T, a.N - j0);
        const float *buf = tbuf(st) + tile_float_offset(cref + size_t(j0) * 3);
        float2 rx[BQ_R / 2], ry[BQ_R / 2], rz[BQ_R / 2];
#pragma unroll
        for (int p = 0; p < BQ_R / 2; ++p) {
            const float *p0 = buf + 3 * (lane + 32 * (2 * p));
            const float *p1 = buf + 3 * (lane + 32 * (2 * p + 1));
            rx[p] = make_float2(p0[0], p1[0]);
            ry[p] = make_float2(p0[1], p1[1]);
            rz[p] = make_float2(p0[2], p1[2]);
        }
        // buffer `st` fully read; stop when every query of the block is full
        const bool all_done = __syncthreads_and(ndone == nq);
        if (*s_err) {
            failed_it = it;
            break;
        }
        if (all_done) {
            stop_it = it;
            break;
        }
        if (threadIdx.x == 0 && it + 2 < a.ntiles) {
            const int j2 = (it + 2) * BQ_T;
            issue_tile(tbuf(st), cref + size_t(j2) * 3, min(BQ_T, a.N - j2),
                       &bars[st]);
        }
        for (int g = 0; g < nq; ++g) {
            const float4 q = qst[g];
            int hits = __float_as_int(q.w);
            if (hits >= K) continue;
            const float2 nx = make_float2(-q.x, -q.x);
            const float2 ny = make_float2(-q.y, -q.y);
            const float2 nz = make_float2(-q.z, -q.z);
            float s[BQ_R];
            bool any = false;
#pragma unroll
            for (int p = 0; p < BQ_R / 2; ++p) {
                const float2 sv = sqdist2(rx[p], ry[p], rz[p], nx, ny, nz, nz0);
                s[2 * p] = sv.x;
                s[2 * p + 1] = sv.y;
                any |= (sv.x < a.R2) | (sv.y < a.R2);
            }
            if (!__any_sync(FULL, any)) continue;
            const size_t row = size_t(b) * a.Q + q_warp0 + g;
#pragma unroll
            for (int r = 0; r < BQ_R; ++r) {
                const bool hit = (r * 32 + lane < cnt) && s[r] < a.R2;
                const unsigned bal = __ballot_sync(FULL, hit);
                if (bal) {
                    const int pos = hits + __popc(bal & lanemask_lt());
                    if (hit && pos < K) {
                        a.out_idx[row * K + pos] = j0 + r * 32 + lane;
                        a.out_dist2[row * K + pos] = s[r];
                    }
                    hits += __popc(bal);
                    if (hits >= K) break;
                }
            }
            hits = min(hits, K);
            if (lane == 0) qst[g].w = __int_as_float(hits);
            if (hits >= K) ++ndone;
        }
    }

    if (threadIdx.x == 0) {
        // let copies still in flight land before the block's shared memory is
        // released: after a stop at tile `it`, tile it + 1 may be in flight
        // (tile it + 2 was never issued)
        const int from = failed_it >= 0 ? failed_it : stop_it;
        for (int it = from; it < from + 2 && it < a.ntiles; ++it)
            if (it > from || failed_it >= 0)
                mbar_wait_bounded(&bars[it & 1], (it >> 1) & 1, a.timeout_ns);
    }
    if (failed_it >= 0) raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);

    // pad the unused slots with (-1, 0)
    __syncwarp();
    for (int g = 0; g < nq; ++g) {
        const size_t row = size_t(b) * a.Q + q_warp0 + g;
        const int hits = failed_it >= 0 ? 0 : __float_as_int(qst[g].w);
        for (int e = hits + lane; e < K; e += 32) {
            a.out_idx[row * K + e] = -1;
            a.out_dist2[row * K + e] = 0.0f;
        }
    }
}

}  // namespace

cudaError_t launch_ball_query(const DeviceInfo &dev, const float *query,
                              int64_t B, int64_t Q, const float *ref,
                              int64_t N, float r32, int64_t K,
                              float *out_dist2, int64_t *out_idx,
                              cudaStream_t stream) {
    BqArgs a{};
    a.query = query;
    a.ref = ref;
    a.Q = static_cast<int>(Q);
    a.N = static_cast<int>(N);
    a.R2 = r32 * r32;  // fl32(fl32(r) * fl32(r)): a single float multiply
    a.K = static_cast<int>(K);
    a.ntiles = static_cast<int>((N + BQ_T - 1) / BQ_T);
    a.out_dist2 = out_dist2;
    a.out_idx = out_idx;
    a.status = dev.status_word;
    a.timeout_ns = wait_timeout_ns();
    a.negzero = -0.0f;

    const int slots = dev.sm_count * 2;
    const int64_t bpc_target = std::max<int64_t>(1, slots / std::max<int64_t>(B, 1));
    int64_t G = (Q + BQ_WARPS * bpc_target - 1) / (BQ_WARPS * bpc_target);
    const size_t budget =
        std::min<size_t>(dev.smem_per_block_optin, dev.smem_per_sm / 2 - 2048);
    const int64_t gmax = std::max<int64_t>(
        1, int64_t((budget - bq_fixed_smem()) / (BQ_WARPS * sizeof(float4))));
    G = std::max<int64_t>(1, std::min(G, gmax));
    a.q_per_warp = static_cast<int>(G);
    const int64_t bpc = (Q + BQ_WARPS * G - 1) / (BQ_WARPS * G);
    const size_t smem = bq_fixed_smem() + size_t(BQ_WARPS) * G * sizeof(float4);
    cudaError_t e = cudaFuncSetAttribute(
        bq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(bpc), static_cast<unsigned>(B));
    bq_kernel<<<grid, BQ_THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pcn
