// pc_knn.cu -- exact brute-force k nearest neighbors on sm_103a.
//
// Operator (mps-pointops project page, "k nearest neighbors"; "Numerical
// contracts", "Selection and output"): for every query, the k references
// that come first in (s, j) order -- squared distance, then index -- with
// D = sqrt(s).
//
// Design (one launch, no scratch memory):
//  * A block of KNN_WARPS warps owns KNN_WARPS * G queries of one cloud; each
//    warp owns G of them.  The warp's queries live in shared memory as
//    float4 (x, y, z, tau) where tau is the query's current k-th squared
//    distance.
//  * Reference tiles of KNN_T = 32 * KNN_R points are staged into shared
//    memory by TMA bulk copies (double buffered, mbarrier completion) and
//    then held in registers: lane l holds tile points l + 32 r, r < KNN_R,
//    packed in pairs for the f32x2 distance instructions.
//  * For each (query, tile) a lane evaluates KNN_R distances (4 packed
//    instructions per pair of references), compares them with tau and one
//    warp vote decides whether any lane has a candidate.  Candidates are rare
//    once a query's list is full.
//  * Each query's sorted list of 32 * KPL (s, j) entries is spread over the
//    warp (lane l holds entries l, l + 32, ...).  A candidate is inserted with
//    one ballot per 32 entries for its rank and a shuffle shift; the order is
//    the lexicographic (s, j) order, so the result does not depend on the
//    order in which tiles are visited.
//  * Tiles are visited in a scrambled order (stride ~0.618 * tiles, coprime
//    with the tile count) so that spatially sorted inputs do not feed each
//    query a stream of ever-closer candidates (the project page's kNN kernel
//    notes reports a 6-8x slowdown from storage order on sorted input).
#include "pc_device.cuh"
#include "pc_internal.h"
#include "pc_tiles.cuh"

#include <algorithm>
#include <climits>

namespace pcn {
namespace {

constexpr int KNN_R = 8;               // reference points per lane per tile
constexpr int KNN_T = 32 * KNN_R;      // reference points per tile
constexpr int KNN_WARPS = 8;           // warps per block
constexpr int KNN_THREADS = 32 * KNN_WARPS;
constexpr unsigned FULL = 0xffffffffu;

struct KnnArgs {
    const float *query;
    const float *ref;
    int Q, N, k;
    int q_per_warp;
    int ntiles, tile_stride;
    float *out_dist;
    int64_t *out_idx;
    int *status;
    uint64_t timeout_ns;
    float negzero;  // -0.0f, see sq2_rn
};

__host__ __device__ constexpr size_t knn_fixed_smem() {
    return 2 * size_t(tile_buffer_bytes(KNN_T)) + 32;
}

__device__ __forceinline__ int knn_tile_at(const KnnArgs &a, int it) {
    return static_cast<int>((static_cast<long long>(it) * a.tile_stride) %
                            a.ntiles);
}

// Entry k-1 of the warp-distributed list: (s, j) broadcast to every lane.
template <int KPL>
__device__ __forceinline__ void list_kth(const float (&ls)[KPL],
                                         const int (&lj)[KPL], int k,
                                         float &ts, int &tj) {
    const int kc = (k - 1) >> 5, kl = (k - 1) & 31;
    float vs = ls[0];
    int vj = lj[0];
#pragma unroll
    for (int c = 1; c < KPL; ++c)
        if (c == kc) {
            vs = ls[c];
            vj = lj[c];
        }
    ts = __shfl_sync(FULL, vs, kl);
    tj = __shfl_sync(FULL, vj, kl);
}

// Insert every candidate of this tile into the query's list.  s[r] is this
// lane's squared distance to tile point r*32 + lane; j0 the tile's first
// index; cnt the number of valid points in the tile.  Warp-uniform.
template <int KPL>
__device__ __forceinline__ void knn_insert(const float (&s)[KNN_R], int j0,
                                        int cnt, int k, float *ls_sm,
                                        int *lj_sm, float *tau_sm) {
    const int lane = static_cast<int>(lane_id());
    float ls[KPL];
    int lj[KPL];
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
        ls[c] = ls_sm[c * 32 + lane];
        lj[c] = lj_sm[c * 32 + lane];
    }
    float ts;
    int tj;
    list_kth<KPL>(ls, lj, k, ts, tj);
    bool changed = false;
#pragma unroll
    for (int r = 0; r < KNN_R; ++r) {
        const int jr = j0 + r * 32 + lane;
        const bool valid = r * 32 + lane < cnt;
        const bool pass = valid && (s[r] < ts || (s[r] == ts && jr < tj));
        unsigned bal = __ballot_sync(FULL, pass);
        while (bal) {
            const int src = __ffs(bal) - 1;
            bal &= bal - 1;
            const float cs = __shfl_sync(FULL, s[r], src);
            const int cj = j0 + r * 32 + src;
            if (cs < ts || (cs == ts && cj < tj)) {
                int pos = 0;
#pragma unroll
                for (int c = 0; c < KPL; ++c)
                    pos += __popc(__ballot_sync(
                        FULL, ls[c] < cs || (ls[c] == cs && lj[c] < cj)));
#pragma unroll
                for (int c = KPL - 1; c >= 0; --c) {
                    float us = __shfl_up_sync(FULL, ls[c], 1);
                    int uj = __shfl_up_sync(FULL, lj[c], 1);
                    if (c > 0) {
                        const float ps = __shfl_sync(FULL, ls[c - 1], 31);
                        const int pj = __shfl_sync(FULL, lj[c - 1], 31);
                        if (lane == 0) {
                            us = ps;
                            uj = pj;
                        }
                    }
                    const int e = c * 32 + lane;
                    if (e > pos) {
                        ls[c] = us;
                        lj[c] = uj;
                    } else if (e == pos) {
                        ls[c] = cs;
                        lj[c] = cj;
                    }
                }
                list_kth<KPL>(ls, lj, k, ts, tj);
                changed = true;
            }
        }
    }
    if (changed) {
#pragma unroll
        for (int c = 0; c < KPL; ++c) {
            ls_sm[c * 32 + lane] = ls[c];
            lj_sm[c * 32 + lane] = lj[c];
        }
        if (lane == 0) *tau_sm = ts;
    }
}

template <int KPL>
__global__ void __launch_bounds__(KNN_THREADS, 2) knn_kernel(const KnnArgs a) {
    constexpr int L = 32 * KPL;
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const float2 nz0 = make_float2(a.negzero, a.negzero);
    const int G = a.q_per_warp;
    const int q_warp0 = (blockIdx.x * KNN_WARPS + warp) * G;
    const int nq = max(0, min(G, a.Q - q_warp0));

    constexpr unsigned BUF = tile_buffer_bytes(KNN_T);
    // tile buffer of stage st: smem + st * BUF
    auto tbuf = [&](int st) { return reinterpret_cast<float *>(smem + st * BUF); };
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 2 * BUF);
    int *s_err = reinterpret_cast<int *>(smem + 2 * BUF + 16);
    float4 *q_all = reinterpret_cast<float4 *>(smem + knn_fixed_smem());
    float *s_all = reinterpret_cast<float *>(q_all + KNN_WARPS * G);
    int *j_all = reinterpret_cast<int *>(s_all + size_t(KNN_WARPS) * G * L);
    float4 *qst = q_all + warp * G;
    float *lst_s = s_all + size_t(warp) * G * L;
    int *lst_j = j_all + size_t(warp) * G * L;

    const float *cref = a.ref + size_t(b) * size_t(a.N) * 3;
    const float *cq = a.query + size_t(b) * size_t(a.Q) * 3;

    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        *s_err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int g = 0; g < G; ++g) {
        if (lane == 0) {
            float4 v = make_float4(0.f, 0.f, 0.f, __int_as_float(0x7f800000));
            if (g < nq) {
                const float *p = cq + size_t(q_warp0 + g) * 3;
                v.x = p[0];
                v.y = p[1];
                v.z = p[2];
            }
            qst[g] = v;
        }
        for (int e = lane; e < L; e += 32) {
            lst_s[g * L + e] = __int_as_float(0x7f800000);
            lst_j[g * L + e] = INT_MAX;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int it = 0; it < 2 && it < a.ntiles; ++it) {
            const int t = knn_tile_at(a, it);
            const int j0 = t * KNN_T;
            issue_tile(tbuf(it), cref + size_t(j0) * 3, min(KNN_T, a.N - j0),
                       &bars[it]);
        }
    }

    int failed_it = -1;
    for (int it = 0; it < a.ntiles; ++it) {
        const int st = it & 1;
        const unsigned par = (it >> 1) & 1;
        if (!mbar_wait_bounded(&bars[st], par, a.timeout_ns)) *s_err = 1;
        const int t = knn_tile_at(a, it);
        const int j0 = t * KNN_T;
        const int cnt = min(KNN_T, a.N - j0);
        const float *buf = tbuf(st) + tile_float_offset(cref + size_t(j0) * 3);
        float2 rx[KNN_R / 2], ry[KNN_R / 2], rz[KNN_R / 2];
#pragma unroll
        for (int p = 0; p < KNN_R / 2; ++p) {
            const float *p0 = buf + 3 * (lane + 32 * (2 * p));
            const float *p1 = buf + 3 * (lane + 32 * (2 * p + 1));
            rx[p] = make_float2(p0[0], p1[0]);
            ry[p] = make_float2(p0[1], p1[1]);
            rz[p] = make_float2(p0[2], p1[2]);
        }
        __syncthreads();  // buffer `st` fully read by every warp
        if (*s_err) {
            failed_it = it;
            break;
        }
        if (threadIdx.x == 0 && it + 2 < a.ntiles) {
            const int t2 = knn_tile_at(a, it + 2);
            const int j2 = t2 * KNN_T;
            issue_tile(tbuf(st), cref + size_t(j2) * 3, min(KNN_T, a.N - j2),
                       &bars[st]);
        }
        float4 qn = nq > 0 ? qst[0] : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int g = 0; g < nq; ++g) {
            const float4 q = qn;
            if (g + 1 < nq) qn = qst[g + 1];
            const float2 nx = make_float2(-q.x, -q.x);
            const float2 ny = make_float2(-q.y, -q.y);
            const float2 nz = make_float2(-q.z, -q.z);
            float s[KNN_R];
            bool any = false;
#pragma unroll
            for (int p = 0; p < KNN_R / 2; ++p) {
                const float2 sv = sqdist2(rx[p], ry[p], rz[p], nx, ny, nz, nz0);
                s[2 * p] = sv.x;
                s[2 * p + 1] = sv.y;
                any |= (sv.x <= q.w) | (sv.y <= q.w);
            }
            if (__any_sync(FULL, any))
                knn_insert<KPL>(s, j0, cnt, a.k, lst_s + g * L, lst_j + g * L,
                                &qst[g].w);
        }
    }

    if (failed_it >= 0) {
        raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
        if (threadIdx.x == 0) {
            // let the copies still in flight (tiles failed_it, failed_it + 1)
            // land before the block's shared memory is released
            for (int it = failed_it; it < failed_it + 2 && it < a.ntiles; ++it)
                mbar_wait_bounded(&bars[it & 1], (it >> 1) & 1, a.timeout_ns);
        }
        for (int g = 0; g < nq; ++g) {
            const size_t row = size_t(b) * a.Q + q_warp0 + g;
            for (int e = lane; e < a.k; e += 32) a.out_idx[row * a.k + e] = -1;
        }
        return;
    }

    for (int g = 0; g < nq; ++g) {
        const size_t row = size_t(b) * a.Q + q_warp0 + g;
#pragma unroll
        for (int c = 0; c < KPL; ++c) {
            const int e = c * 32 + lane;
            if (e < a.k) {
                a.out_idx[row * a.k + e] = lst_j[g * L + e];
                a.out_dist[row * a.k + e] = __fsqrt_rn(lst_s[g * L + e]);
            }
        }
    }
}

int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// A stride near 0.618 * n that is coprime with n, so that it*stride mod n
// visits every tile once.
int scramble_stride(int n) {
    if (n <= 2) return 1;
    int s = std::max(1, static_cast<int>(0.6180339887 * n));
    while (gcd_int(s, n) != 1) ++s;
    return s % n == 0 ? 1 : s;
}

template <int KPL>
cudaError_t launch_knn_t(const DeviceInfo &dev, const KnnArgs &a0, int64_t B,
                         int64_t Q, cudaStream_t stream) {
    KnnArgs a = a0;
    constexpr int L = 32 * KPL;
    const size_t per_q = sizeof(float4) + size_t(L) * 8;
    const int slots = dev.sm_count * 2;
    // queries per warp: spread B*Q over about one wave of 2 blocks per SM
    const int64_t bpc_target = std::max<int64_t>(1, slots / std::max<int64_t>(B, 1));
    int64_t G = (Q + KNN_WARPS * bpc_target - 1) / (KNN_WARPS * bpc_target);
    const size_t budget =
        std::min<size_t>(dev.smem_per_block_optin, dev.smem_per_sm / 2 - 2048);
    const int64_t gmax = std::max<int64_t>(
        1, int64_t((budget - knn_fixed_smem()) / (KNN_WARPS * per_q)));
    G = std::max<int64_t>(1, std::min(G, gmax));
    a.q_per_warp = static_cast<int>(G);
    const int64_t bpc = (Q + KNN_WARPS * G - 1) / (KNN_WARPS * G);
    const size_t smem = knn_fixed_smem() + size_t(KNN_WARPS) * G * per_q;
    cudaError_t e = cudaFuncSetAttribute(
        knn_kernel<KPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(bpc), static_cast<unsigned>(B));
    knn_kernel<KPL><<<grid, KNN_THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_knn(const DeviceInfo &dev, const float *query, int64_t B,
                       int64_t Q, const float *ref, int64_t N, int k,
                       float *out_dist, int64_t *out_idx,
                       cudaStream_t stream) {
    KnnArgs a{};
    a.query = query;
    a.ref = ref;
    a.Q = static_cast<int>(Q);
    a.N = static_cast<int>(N);
    a.k = k;
    a.ntiles = static_cast<int>((N + KNN_T - 1) / KNN_T);
    a.tile_stride = scramble_stride(a.ntiles);
    a.out_dist = out_dist;
    a.out_idx = out_idx;
    a.status = dev.status_word;
    a.timeout_ns = wait_timeout_ns();
    a.negzero = -0.0f;
    if (k <= 32) return launch_knn_t<1>(dev, a, B, Q, stream);
    if (k <= 64) return launch_knn_t<2>(dev, a, B, Q, stream);
    if (k <= 128) return launch_knn_t<4>(dev, a, B, Q, stream);
    return launch_knn_t<8>(dev, a, B, Q, stream);
}

}  // namespace pcn
