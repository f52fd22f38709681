// pc_knn.cu -- exact brute-force k nearest neighbors on sm_103a.
//
// Operator (mps-pointops project page, "k nearest neighbors"; "Numerical
// contracts", "Selection and output"): for every query, the k references
// that come first in (s, j) order -- squared distance, then index -- with
// D = sqrt(s).
//
// Two kernels.  k <= 32: knn_lane_kernel (below), one or two queries per
// lane with per-lane heaps, fed by a producer warp that prepares the tiles
// (pc_stream.cuh); large clouds are first put in a spatial order (a few
// small kernels and stream-ordered scratch) that the kernel visits outwards
// from each block's region.  k > 32, and launches with too few queries to
// give every SM a warp of the lane kernel: knn_kernel, described here (one
// launch, no scratch memory):
//  * A block has KNN_CWARPS consumer warps and one producer warp.  Consumer
//    warp w owns G queries of one cloud.  Per query, shared memory holds the
//    filter constants (-2q', -2q', thr, thr; pc_filter.cuh), the raw
//    coordinates and |q'|^2, and the query's sorted list of k (s, j) entries.
//  * The producer's lane 0 streams reference tiles of KNN_T = 32 * KNN_R
//    points through a KNN_STAGES ring in shared memory with TMA bulk copies
//    (full/empty mbarriers, see TileRing); consumer warps derive the centred
//    coordinates and w' of their KNN_R points per lane (lane l holds points
//    l + 32 r, packed in pairs) into registers and keep the raw tile in the
//    ring until their queries are done, drifting freely instead of meeting
//    at a block barrier.
//  * Per (query, tile) a lane evaluates the conservative filter of
//    pc_filter.cuh for its KNN_R points (three packed FMAs per pair of
//    points) against the query's threshold; one vote decides whether the
//    warp looks closer.  The hot loop is only those FMAs, the compares and
//    the vote.  Candidates are rare once a list is full.
//  * The slow path computes the exact s32 of the tile's points from the raw
//    coordinates in shared memory; each lane builds a bitmask of its slots
//    that beat the list's k-th (s, j) entry and parks its distances in a
//    per-warp scratch row; the warp walks the candidates and inserts each
//    into the warp-distributed list (lane l holds entries l, l + 32, ...):
//    one ballot per 32 entries gives the rank, a shuffle shift makes room.
//    The order is the lexicographic (s, j) order, so the result does not
//    depend on the order in which candidates or tiles are visited.
//  * Tiles are visited in a scrambled order (stride ~0.618 * tiles, coprime
//    with the tile count) so that spatially sorted inputs do not feed each
//    query a stream of ever-closer candidates (the project page's kNN kernel
//    notes report a 6-8x slowdown from storage order on sorted input).
#include "pointcloud.h"
#include "pc_device.cuh"
#include "pc_filter.cuh"
#include "pc_internal.h"
#include "pc_stream.cuh"
#include "pc_tiles.cuh"

#include <algorithm>
#include <type_traits>
#include <climits>

namespace pcn {
namespace {

constexpr int KNN_R = 8;                  // reference points per lane per tile
constexpr int KNN_T = 32 * KNN_R;         // reference points per tile
constexpr int KNN_CWARPS = 8;             // consumer warps per block
constexpr int KNN_THREADS = 32 * (KNN_CWARPS + 1);
constexpr int KNN_STAGES = 4;
constexpr unsigned FULL = 0xffffffffu;

struct KnnArgs {
    const float *query;
    const float *ref;
    const int64_t *q_len;  // valid queries per cloud (NULL: Q)
    const int64_t *r_len;  // valid references per cloud (NULL: N)
    int Q, N, k;
    int squared;           // return s instead of sqrt(s)
    int q_per_warp;
    float *out_dist;
    int64_t *out_idx;
    int *status;
    uint64_t timeout_ns;
    int stall;  // PC_STALL_* testing flags
    // spatial order (lane kernel, ORDERED): per cloud the valid references
    // and queries as 16-byte points (x, y, z, original index bits) sorted by
    // cell code, the starts of the reference cells and the cell frame
    const float *sref;    // [B][N] x 4
    const float *squery;  // [B][Q] x 4 (== sref for a query set equal to ref)
    const int *cstart;    // [B][MC_CELLS + 1]
    const float *cframe;  // [B][8]: lo x, y, z, scale x, y, z
    // ORDERED with the references split into gridDim.z parts: each part's
    // sorted k keys per valid query row, [part][B][Q][k] (merged afterwards)
    unsigned long long *part_keys;
    // ORDERED: per query (in the query order) the exact k best keys over its
    // seeded tile, as a max-heap [B][Q][k] (knn_seed_kernel)
    const unsigned long long *seed;
    // ORDERED, Ball Query fused in (bq_rows != NULL; one part): per query
    // (in the query order) the bq_K smallest indices j with s32 < bq_R2 seen
    // so far, as (j, s32 bits) in bq_rows [B][Q][bq_K] in no order, and its
    // state in bq_state [B][Q]: (hits seen, largest kept j, its slot, -) --
    // hits -1 when the query's search stopped on a timeout.
    // knn_bq_finish_kernel sorts each row by j into bq_out_*.
    int2 *bq_rows;
    int4 *bq_state;
    float bq_R2;
    int bq_K;
    float *bq_out_d2;
    int64_t *bq_out_idx;
};

// A Ball Query hit (j, s) of a query whose bq_K slots are `row`: the slots
// keep the K smallest indices among all hits seen, in no order; (hits,
// maxj, maxpos) is the query's state (hits seen, largest kept index, its
// slot).  Once K slots are full, a smaller index replaces the largest and the
// slots are scanned for the new largest (a query has that many hits only
// where the cloud is dense).
__device__ __forceinline__ void bq_keep(int2 *row, int K, int &hits, int &maxj,
                                        int &maxpos, int j, float s) {
    if (hits < K) {
        row[hits] = make_int2(j, __float_as_int(s));
        if (j > maxj) {
            maxj = j;
            maxpos = hits;
        }
    } else if (j < maxj) {
        row[maxpos] = make_int2(j, __float_as_int(s));
        maxj = -1;
        for (int e = 0; e < K; ++e) {
            const int je = row[e].x;
            if (je > maxj) {
                maxj = je;
                maxpos = e;
            }
        }
    }
    ++hits;
}

// Cell codes of the spatial order: MC_BITS bits per axis, interleaved
// (Morton order), so that a run of consecutive cells is a compact block.
constexpr int MC_BITS = 5;
constexpr int MC_CELLS = 1 << (3 * MC_BITS);

__device__ __forceinline__ unsigned mc_spread(unsigned v) {  // 5 bits -> every 3rd
    unsigned r = 0;
#pragma unroll
    for (int i = 0; i < MC_BITS; ++i) r |= ((v >> i) & 1u) << (3 * i);
    return r;
}

// Code of (x, y, z) in the frame f (lo, scale); coordinates outside the
// frame or NaN go to the nearest edge cell (any cell is correct: the code
// only orders the points).
__device__ __forceinline__ unsigned mc_code(const float *f, float x, float y, float z) {
    const int hi = (1 << MC_BITS) - 1;
    const int cx = min(hi, max(0, __float2int_rz(__fmul_rn(__fsub_rn(x, f[0]), f[3]))));
    const int cy = min(hi, max(0, __float2int_rz(__fmul_rn(__fsub_rn(y, f[1]), f[4]))));
    const int cz = min(hi, max(0, __float2int_rz(__fmul_rn(__fsub_rn(z, f[2]), f[5]))));
    return mc_spread(unsigned(cx)) | (mc_spread(unsigned(cy)) << 1) |
           (mc_spread(unsigned(cz)) << 2);
}

// One query in shared memory: the filter constants duplicated so that the
// halves are packed operands, and the raw coordinates for the exact path.
struct __align__(16) QuerySlot {
    float4 axy;  // (-2x', -2x', -2y', -2y')   centred coordinates
    float4 azt;  // (-2z', -2z', thr, thr)     filter threshold
    float4 raw;  // (x, y, z, |q'|^2)
    float4 kth;  // (s, j (int bits), -, -) of the list's k-th entry
};

constexpr unsigned KNN_BUF = tile_buffer_bytes(KNN_T);

__host__ __device__ constexpr size_t knn_fixed_smem() {
    // ring, 2 * STAGES mbarriers, error flag, per-warp candidate scratch
    return size_t(KNN_STAGES) * KNN_BUF + 2 * KNN_STAGES * 8 + 16 +
           size_t(KNN_CWARPS) * 32 * KNN_R * sizeof(float);
}

__host__ __device__ constexpr size_t knn_per_query_smem(int k) {
    return sizeof(QuerySlot) + size_t(k) * (sizeof(float) + sizeof(int));
}

__device__ __forceinline__ int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// A stride near 0.618 * n that is coprime with n, so that it*stride mod n
// visits every tile once (the project page's scrambled chunk order).
__device__ __forceinline__ int scramble_stride(int n) {
    if (n <= 2) return 1;
    int s = max(1, static_cast<int>(0.6180339887 * n));
    while (gcd_int(s, n) != 1) ++s;
    return s % n == 0 ? 1 : s;
}

__device__ __forceinline__ int knn_tile_at(int it, int stride, int ntiles) {
    return static_cast<int>((static_cast<long long>(it) * stride) % ntiles);
}

// Valid length of cloud b: lens[b] clamped to [0, full], or full.
__device__ __forceinline__ int valid_len(const int64_t *lens, int b, int full) {
    if (lens == nullptr) return full;
    const int64_t v = lens[b];
    return v < 0 ? 0 : (v > full ? full : static_cast<int>(v));
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

// Insert this tile's candidates for one query (warp-uniform), called when
// the filter let at least one pair through.  The lane's filter mask is
// recomputed from its registers; only points that pass get their exact s32
// (from the raw tile in shared memory, lane l: points l + 32 r), and only
// those that beat the list's k-th (s, j) entry are inserted.  The list is
// not touched when every pass was a false positive.
template <int KPL>
__device__ __forceinline__ void knn_insert(const float *tile,
                                           const float2 (&rx)[KNN_R / 2],
                                           const float2 (&ry)[KNN_R / 2],
                                           const float2 (&rz)[KNN_R / 2],
                                           const float2 (&rw)[KNN_R / 2],
                                           float4 axy, float4 azt, int j0,
                                           int cnt, int k, QuerySlot *qs,
                                           float *ls_sm, int *lj_sm,
                                           float *scratch) {
    const int lane = static_cast<int>(lane_id());
    unsigned pm = filter_mask8(rx, ry, rz, rw, axy, azt);
    const int left = cnt - lane;  // points r with r * 32 < left are valid
    pm &= left >= KNN_T ? 0xffu : (left > 0 ? (1u << ((left + 31) >> 5)) - 1u : 0u);
    const float4 q = qs->raw;
    const float4 kth = qs->kth;
    float ts = kth.x;
    int tj = __float_as_int(kth.y);
    unsigned m = 0;
    while (pm) {
        const int r = __ffs(pm) - 1;
        pm &= pm - 1;
        const float *p = tile + 3 * (lane + 32 * r);
        const float sv = sqdist(q.x, q.y, q.z, p[0], p[1], p[2]);
        const int j = j0 + r * 32 + lane;
        if (sv < ts || (sv == ts && j < tj)) {
            m |= 1u << r;
            scratch[lane * KNN_R + r] = sv;
        }
    }
    unsigned bal = __ballot_sync(FULL, m != 0);
    if (bal == 0) return;
    float ls[KPL];
    int lj[KPL];
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
        const int e = c * 32 + lane;
        ls[c] = e < k ? ls_sm[e] : __int_as_float(0x7f800000);
        lj[c] = e < k ? lj_sm[e] : INT_MAX;
    }
    __syncwarp();
    while (bal) {
        const int src = __ffs(bal) - 1;
        bal &= bal - 1;
        unsigned mm = __shfl_sync(FULL, m, src);
        while (mm) {
            const int r = __ffs(mm) - 1;
            mm &= mm - 1;
            const float cs = scratch[src * KNN_R + r];
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
            }
        }
    }
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
        const int e = c * 32 + lane;
        if (e < k) {
            ls_sm[e] = ls[c];
            lj_sm[e] = lj[c];
        }
    }
    if (lane == 0) {
        const float thr = tj == INT_MAX ? __int_as_float(0x7f800000)
                                        : filter_threshold(ts, q.w);
        qs->azt.z = thr;
        qs->azt.w = thr;
        qs->kth = make_float4(ts, __int_as_float(tj), 0.f, 0.f);
    }
    __syncwarp();  // the scratch row is reused by the next insertion
}

template <int KPL>
__global__ void __launch_bounds__(KNN_THREADS, 2) knn_kernel(const KnnArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int G = a.q_per_warp;
    const int k = a.k;

    TileRing ring;
    ring.base = smem;
    ring.bytes = KNN_BUF;
    ring.full = reinterpret_cast<uint64_t *>(smem + KNN_STAGES * KNN_BUF);
    ring.empty = ring.full + KNN_STAGES;
    int *s_err = reinterpret_cast<int *>(ring.empty + KNN_STAGES);
    float *scratch_all = reinterpret_cast<float *>(
        smem + KNN_STAGES * KNN_BUF + 2 * KNN_STAGES * 8 + 16);
    QuerySlot *slots_all =
        reinterpret_cast<QuerySlot *>(smem + knn_fixed_smem());
    float *ls_all = reinterpret_cast<float *>(slots_all + KNN_CWARPS * G);
    int *lj_all = reinterpret_cast<int *>(ls_all + size_t(KNN_CWARPS) * G * k);

    const float *cref = a.ref + size_t(b) * size_t(a.N) * 3;
    const int Nb = valid_len(a.r_len, b, a.N);
    const int Qb = valid_len(a.q_len, b, a.Q);
    const int ntiles = (Nb + KNN_T - 1) / KNN_T;
    const int tstride = scramble_stride(ntiles);

    if (blockIdx.x * KNN_CWARPS * G >= Qb) {
        // every query of this block is past the cloud's valid length
        const int r0 = blockIdx.x * KNN_CWARPS * G;
        const int r1 = min(a.Q, r0 + KNN_CWARPS * G);
        const size_t e0 = (size_t(b) * a.Q + r0) * k;
        const size_t e1 = (size_t(b) * a.Q + r1) * k;
        for (size_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
            a.out_idx[e] = -1;
            a.out_dist[e] = 0.0f;
        }
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < KNN_STAGES; ++s) {
            mbar_init(&ring.full[s], 1);
            mbar_init(&ring.empty[s], KNN_CWARPS);
        }
        *s_err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }

    if (warp == KNN_CWARPS) {  // producer warp
        __syncthreads();
        const bool withhold = (a.stall & PC_STALL_TILE_STREAM) && blockIdx.x == 0 &&
                              blockIdx.y == 0;
        if (lane == 0)
            ring_produce<KNN_STAGES>(
                ring, cref, Nb, KNN_T, ntiles,
                [&](int it) { return knn_tile_at(it, tstride, ntiles); }, s_err,
                s_err, a.timeout_ns, withhold);
        return;
    }

    // consumer warp: set up this warp's queries and lists
    const int q_warp0 = (blockIdx.x * KNN_CWARPS + warp) * G;
    const int nq = max(0, min(G, Qb - q_warp0));
    QuerySlot *slots = slots_all + warp * G;
    float *ls_w = ls_all + size_t(warp) * G * k;
    int *lj_w = lj_all + size_t(warp) * G * k;
    float *scratch = scratch_all + warp * 32 * KNN_R;
    const float *cq = a.query + size_t(b) * size_t(a.Q) * 3;
    const float inf = __int_as_float(0x7f800000);
    const FilterFrame fr = filter_frame(cref, min(KNN_T, Nb));
    for (int g = lane; g < G; g += 32) {
        float x = 0.f, y = 0.f, z = 0.f;
        if (g < nq) {
            const float *p = cq + size_t(q_warp0 + g) * 3;
            x = p[0];
            y = p[1];
            z = p[2];
        }
        const float xp = __fsub_rn(x, fr.cx), yp = __fsub_rn(y, fr.cy),
                    zp = __fsub_rn(z, fr.cz);
        float ax, ay, az;
        const float qq = filter_query(xp, yp, zp, ax, ay, az);
        slots[g].axy = make_float4(ax, ax, ay, ay);
        slots[g].azt = make_float4(az, az, inf, inf);
        slots[g].raw = make_float4(x, y, z, qq);
        slots[g].kth = make_float4(inf, __int_as_float(INT_MAX), 0.f, 0.f);
    }
    for (int e = lane; e < G * k; e += 32) {
        ls_w[e] = inf;
        lj_w[e] = INT_MAX;
    }
    __syncthreads();

    bool failed = false;
    for (int it = 0; it < ntiles; ++it) {
        const int st = it % KNN_STAGES;
        const WaitResult w = mbar_wait_or_stop(
            &ring.full[st], unsigned((it / KNN_STAGES) & 1), s_err, a.timeout_ns);
        if (!__all_sync(FULL, w == WAIT_OK)) {
            failed = true;
            break;
        }
        const int j0 = knn_tile_at(it, tstride, ntiles) * KNN_T;
        const int cnt = min(KNN_T, Nb - j0);
        const float *buf =
            ring.buf(st) + tile_float_offset(cref + size_t(j0) * 3);
        // centred coordinates and w' of this lane's points (points past cnt
        // hold stale values: they may pass the filter and are masked exactly)
        float2 rx[KNN_R / 2], ry[KNN_R / 2], rz[KNN_R / 2], rw[KNN_R / 2];
#pragma unroll
        for (int p = 0; p < KNN_R / 2; ++p) {
            const float *p0 = buf + 3 * (lane + 32 * (2 * p));
            const float *p1 = buf + 3 * (lane + 32 * (2 * p + 1));
            float x0 = __fsub_rn(p0[0], fr.cx), y0 = __fsub_rn(p0[1], fr.cy),
                  z0 = __fsub_rn(p0[2], fr.cz);
            float x1 = __fsub_rn(p1[0], fr.cx), y1 = __fsub_rn(p1[1], fr.cy),
                  z1 = __fsub_rn(p1[2], fr.cz);
            const float w0 = filter_ref(x0, y0, z0), w1 = filter_ref(x1, y1, z1);
            rx[p] = make_float2(x0, x1);
            ry[p] = make_float2(y0, y1);
            rz[p] = make_float2(z0, z1);
            rw[p] = make_float2(w0, w1);
        }

        // two queries per step: independent filter chains for the scheduler
        int g = 0;
        for (; g + 1 < nq; g += 2) {
            QuerySlot *s0 = slots + g;
            const float4 axy0 = s0[0].axy, azt0 = s0[0].azt;
            const float4 axy1 = s0[1].axy, azt1 = s0[1].azt;
            const bool t0 = filter_any8(rx, ry, rz, rw, axy0, azt0);
            const bool t1 = filter_any8(rx, ry, rz, rw, axy1, azt1);
            const bool v0 = __any_sync(FULL, t0), v1 = __any_sync(FULL, t1);
            if (v0)
                knn_insert<KPL>(buf, rx, ry, rz, rw, axy0, azt0, j0, cnt, k, s0,
                                ls_w + size_t(g) * k, lj_w + size_t(g) * k, scratch);
            if (v1)
                knn_insert<KPL>(buf, rx, ry, rz, rw, axy1, azt1, j0, cnt, k, s0 + 1,
                                ls_w + size_t(g + 1) * k, lj_w + size_t(g + 1) * k,
                                scratch);
        }
        if (g < nq) {
            QuerySlot *s0 = slots + g;
            const float4 axy = s0->axy, azt = s0->azt;
            if (__any_sync(FULL, filter_any8(rx, ry, rz, rw, axy, azt)))
                knn_insert<KPL>(buf, rx, ry, rz, rw, axy, azt, j0, cnt, k, s0,
                                ls_w + size_t(g) * k, lj_w + size_t(g) * k, scratch);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[st]);  // raw tile no longer read
    }

    // rows of this warp past the valid length: padding
    const int nrows = max(0, min(G, a.Q - q_warp0));
    for (int g = nq; g < nrows; ++g) {
        const size_t row = size_t(b) * a.Q + q_warp0 + g;
        for (int e = lane; e < k; e += 32) {
            a.out_idx[row * k + e] = -1;
            a.out_dist[row * k + e] = 0.0f;
        }
    }
    if (failed) {
        if (lane == 0) *s_err = 1;
        raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
        for (int g = 0; g < nq; ++g) {
            const size_t row = size_t(b) * a.Q + q_warp0 + g;
            for (int e = lane; e < k; e += 32) a.out_idx[row * k + e] = -1;
        }
        return;
    }
    // slots past the number of valid references (k > Nb): padding
    const int kv = min(k, Nb);
    for (int g = 0; g < nq; ++g) {
        const size_t row = size_t(b) * a.Q + q_warp0 + g;
        for (int e = lane; e < k; e += 32) {
            const float sv = ls_w[g * k + e];
            a.out_idx[row * k + e] = e < kv ? int64_t(lj_w[g * k + e]) : int64_t(-1);
            a.out_dist[row * k + e] =
                e < kv ? (a.squared ? sv : __fsqrt_rn(sv)) : 0.0f;
        }
    }
}

// ---------------------------------------------------------------------------
// k <= 32: a lane owns one or two queries (the kernel used for every k up to
// 32).
//
// The producer warp streams the tiles (scrambled order, or outwards from the
// block's home tile in the spatial order) and prepares them
// (pc_stream.cuh).  A lane keeps each query's current k best (s, j) as a
// max-heap of 64-bit keys in shared memory (entry e of lane l at
// [e * 32 + l], root = the k-th best) and the query's filter threshold in a
// register, following the root.  Pass 1, per tile: each 8-point step is
// filtered (three packed FMAs per two points, broadcast shared-memory
// operands) and sets one bit of a pending mask when anything passes.  Pass
// 2: while any lane has a pending step, each such lane re-filters one,
// takes the exact s32 of the points that pass from the stage's raw copy and
// replaces the root by every point that beats it (sift-down).  At the end
// each lane heap-sorts its k keys into ascending (s, j) order.
// ---------------------------------------------------------------------------
// QL queries per lane: 2 for k <= 16, 1 above.  A warp owns a group of
// 32 * QL consecutive queries.
//
// Work layout: one block per SM and wave, with W consumer warps chosen so
// that every SM gets about the same number of query groups (W = ceil(groups
// / (SMs x waves))); warp w of block x owns group w * gridDim.x + x of its
// cloud, so a block's groups are spread over the cloud and the blocks of a
// launch differ by at most one group.  (Blocks of a fixed 256 queries left
// 100k queries at 2.57 blocks per SM against 3 slots: the SMs with three
// blocks set the time.)  ORDERED, a block takes upb consecutive units of 32
// queries instead (upb = ceil(units / (SMs x waves))), so that with two
// slots per lane the SMs differ by half a warp, not a warp: 100k queries on
// 152 SMs are 149 blocks of 10.5 warps' work where 143 blocks of 11 were
// (GB300, k = 16: 2.06 -> 2.01 ms).  One producer serves all W consumer warps.
// consumer warps per block at most (one block per SM: registers)
__host__ __device__ constexpr int kl_wmax(int QL) { return QL == 1 ? 15 : 12; }

__host__ __device__ constexpr size_t knn_lane_smem(int k, int QL, int W) {
    return stream_smem_bytes() + size_t(W) * 32 * QL * size_t(k) * 8;
}

// A heap entry (s, j) as one 64-bit key: the bits of s (a squared distance:
// +0 .. +inf, never NaN in a heap) above j (0 .. INT_MAX).  For such s the
// float order is the order of the bit patterns, so the unsigned order of the
// keys is the lexicographic (s, j) order.  The empty entry is (+inf, INT_MAX).
__device__ __forceinline__ unsigned long long sj_key(float s, int j) {
    return (static_cast<unsigned long long>(__float_as_uint(s)) << 32) |
           static_cast<unsigned>(j);
}
__device__ __forceinline__ float key_s(unsigned long long key) {
    return __uint_as_float(static_cast<unsigned>(key >> 32));
}
__device__ __forceinline__ int key_j(unsigned long long key) {
    return static_cast<int>(static_cast<unsigned>(key));
}
constexpr unsigned long long KEY_EMPTY = 0x7f8000007fffffffull;
// A part that stopped on a device timeout marks its rows with this key (above
// every real or empty key); the merge then writes the row as -1.
constexpr unsigned long long KEY_FAILED = ~0ull;

// Sift `key` down from `pos` in the max-heap h of n keys (stride 32);
// returns the key then at `pos`.
__device__ __forceinline__ unsigned long long heap_sift(unsigned long long *h, int n,
                                                        int pos,
                                                        unsigned long long key) {
    unsigned long long top = key;
    bool first = true;
    for (;;) {
        int c = 2 * pos + 1;
        if (c >= n) break;
        unsigned long long ck = h[c * 32];
        if (c + 1 < n) {
            const unsigned long long dk = h[(c + 1) * 32];
            if (dk > ck) {
                ++c;
                ck = dk;
            }
        }
        if (ck <= key) break;
        h[pos * 32] = ck;
        if (first) top = ck;
        first = false;
        pos = c;
    }
    h[pos * 32] = key;
    return top;
}

// ORDERED: the place among the references of the query at position qpos of
// the query order: qpos itself when the query set is the reference set, else
// the start of its cell.
__device__ __forceinline__ int seed_pos(const KnnArgs &a, int b, int qpos, float qx,
                                        float qy, float qz) {
    const bool self = a.squery == a.sref && a.Q == a.N && a.q_len == a.r_len;
    return self ? qpos
                : a.cstart[size_t(b) * (MC_CELLS + 1) +
                           mc_code(a.cframe + size_t(b) * 8, qx, qy, qz)];
}

// ORDERED: the reference tile seeded for that query, the tile of its place;
// -1 without references.  (Seeding the two tiles next to it as well
// measured slower at 100k points, k = 16: 2.21 vs 2.11 ms.)
__device__ __forceinline__ int seed_tile(const KnnArgs &a, int b, int qpos, float qx,
                                         float qy, float qz, int ntiles) {
    return min(seed_pos(a, b, qpos, qx, qy, qz) / ST_T, ntiles - 1);
}

// ORDERED: one thread per valid query: the exact k best (s, j) over its
// seeded tile (up to ST_T references), kept as a max-heap of keys in
// shared memory (entry e of a warp's lane l at [e * 32 + l]) and written out
// as it stands.  The tile is read outwards from the query's own place
// (o, o - 1, o + 1, o - 2, ..., then the rest of the longer side): in the
// spatial order the nearest references come first, so the heap root falls
// early and few later references need a sift.  The heap holds the k
// smallest keys whatever the order.  Lanes of a warp hold neighbouring
// queries, so they read neighbouring references.
constexpr int SEED_THREADS = 256;
constexpr int SEED_UNROLL = 4;

__global__ void __launch_bounds__(SEED_THREADS) knn_seed_kernel(const KnnArgs a,
                                                                unsigned long long *seed) {
    extern __shared__ __align__(16) unsigned long long seed_heaps[];
    const int b = blockIdx.y;
    const int i = blockIdx.x * SEED_THREADS + threadIdx.x;
    const int Qb = valid_len(a.q_len, b, a.Q);
    if (i >= Qb) return;
    const int k = a.k;
    const int Nb = valid_len(a.r_len, b, a.N);
    const int ntiles = (Nb + ST_T - 1) / ST_T;
    unsigned long long *h = seed_heaps + size_t(threadIdx.x >> 5) * 32 * k + (threadIdx.x & 31);
    for (int e = 0; e < k; ++e) h[e * 32] = KEY_EMPTY;
    const float4 qv = reinterpret_cast<const float4 *>(a.squery)[size_t(b) * a.Q + i];
    const int pos = seed_pos(a, b, i, qv.x, qv.y, qv.z);
    const int t = min(pos / ST_T, ntiles - 1);  // as seed_tile
    const float4 *rp = reinterpret_cast<const float4 *>(a.sref) + size_t(b) * a.N;
    unsigned long long root = KEY_EMPTY;
    const int jlo = max(t, 0) * ST_T;
    const int j1 = min(Nb, (t + 1) * ST_T);
    const int cnt = j1 - jlo;  // 0 without references
    // visit m of the tile -> reference: alternately right (from o) and left
    // (from o - 1) while both sides last, then the longer side on its own
    const int o = min(max(pos, jlo), j1 - 1);
    const int L = o - jlo, R = j1 - o, mm = min(L, R);
    auto ref_at = [&](int m) {
        if (m < 2 * mm) return (m & 1) ? o - 1 - (m >> 1) : o + (m >> 1);
        const int rem = m - 2 * mm;
        return R > L ? o + mm + rem : o - 1 - mm - rem;
    };
    // Ball Query fused in: this tile's hits (the lane kernel skips the tile)
    const bool bq = a.bq_rows != nullptr;
    int2 *bq_row = bq ? a.bq_rows + (size_t(b) * a.Q + i) * a.bq_K : nullptr;
    int bq_hits = 0, bq_maxj = -1, bq_maxpos = 0;
    int m = 0;
    // SEED_UNROLL references at a time: their loads and distances are
    // independent
    for (; m + SEED_UNROLL <= cnt; m += SEED_UNROLL) {
        unsigned long long key[SEED_UNROLL];
#pragma unroll
        for (int u = 0; u < SEED_UNROLL; ++u) {
            const float4 r = rp[ref_at(m + u)];
            const float s = sqdist(qv.x, qv.y, qv.z, r.x, r.y, r.z);
            // s32 >= +0; a NaN s32 has a key above KEY_EMPTY: never taken
            key[u] = sj_key(s, __float_as_int(r.w));
            if (bq && s < a.bq_R2)
                bq_keep(bq_row, a.bq_K, bq_hits, bq_maxj, bq_maxpos, __float_as_int(r.w), s);
        }
#pragma unroll
        for (int u = 0; u < SEED_UNROLL; ++u)
            if (key[u] < root) root = heap_sift(h, k, 0, key[u]);
    }
    for (; m < cnt; ++m) {
        const float4 r = rp[ref_at(m)];
        const float s = sqdist(qv.x, qv.y, qv.z, r.x, r.y, r.z);
        const unsigned long long key = sj_key(s, __float_as_int(r.w));
        if (bq && s < a.bq_R2)
            bq_keep(bq_row, a.bq_K, bq_hits, bq_maxj, bq_maxpos, __float_as_int(r.w), s);
        if (key < root) root = heap_sift(h, k, 0, key);
    }
    unsigned long long *out = seed + (size_t(b) * a.Q + i) * k;
    for (int e = 0; e < k; ++e) out[e] = h[e * 32];
    if (bq) a.bq_state[size_t(b) * a.Q + i] = make_int4(bq_hits, bq_maxj, bq_maxpos, 0);
}

// Pass 1 over one prepared tile for the first NQ query slots of a lane: per
// 8-point step and query, the filter of the step's points (three packed FMAs
// per pair), their minimum and one compare set the step's bit of pend[q].
// Rows of 2^KL_SB steps with compile-time slot offsets (the stage swizzle).
template <int NQ, int KL_QL, int KL_SB>
__device__ __forceinline__ void lane_pass1(const float4 *ck, int nsteps,
                                           const float2 (&ax)[KL_QL],
                                           const float2 (&ay)[KL_QL],
                                           const float2 (&az)[KL_QL],
                                           const float (&thr)[KL_QL],
                                           unsigned (&pend)[KL_QL]) {
    constexpr int KL_ROW = 1 << KL_SB;
    static_assert(8 % KL_ROW == 0, "rows of steps divide 8");
    for (int s0 = 0; s0 < nsteps; s0 += KL_ROW) {
#pragma unroll
        for (int ss = 0; ss < KL_ROW; ++ss) {
            const int step = s0 + ss;
            const float4 *row = ck + 8 * step;
            const int x = ss << (3 - KL_SB);  // the row's slot swizzle
            float mn[NQ];  // running min of t' over the step's points
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 A = row[(2 * u) ^ x];
                const float4 Z = row[(2 * u + 1) ^ x];
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    float2 v = __ffma2_rn(make_float2(A.x, A.y), ax[q],
                                          make_float2(Z.z, Z.w));
                    v = __ffma2_rn(make_float2(A.z, A.w), ay[q], v);
                    v = __ffma2_rn(make_float2(Z.x, Z.y), az[q], v);
                    mn[q] = u == 0 ? fminf(v.x, v.y) : fmin3(mn[q], v.x, v.y);
                }
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) pend[q] |= (mn[q] <= thr[q] ? 1u : 0u) << step;
        }
    }
}

// Two problems with the same k can share one launch: block rows
// blockIdx.y < B0 run a0 (cloud blockIdx.y), the rest a1 (cloud
// blockIdx.y - B0) -- used for the two directions of the Chamfer distance.
//
// ORDERED: the clouds come in the spatial order of the cell codes (sref,
// squery); a block owns `upb` consecutive units of 32 queries (a compact
// region; warp w takes units w * KL_QL .. w * KL_QL + KL_QL - 1 of them) and
// visits the reference tiles outwards from the tile where its region's
// middle query would sit (home, home + 1, home - 1, ...), so the k best
// (s, j) are found in the first few tiles and the later tiles rarely let a
// pair through.  With two slots per lane an odd `upb` leaves the last warp
// one unit: it runs the tile loop for one query per lane, pass 1 at about
// half the cost, so the launch can balance the SMs to half a warp.  Keys
// carry the original indices, so the result is that of the input order.
//
// BQ (ORDERED, one part): Ball Query of the same queries and references in
// the same pass.  Its filter bound is R2, so a query's threshold is the
// larger of its kNN bound and R2's; in pass 2 every exact s32 goes to both
// rules (heap insertion for kNN, s32 < R2 for Ball Query, whose hits are
// kept with bq_keep from the state left by knn_seed_kernel).
template <int KL_QL, bool ORDERED, bool BQ = false>
__global__ void __launch_bounds__(32 * (kl_wmax(KL_QL) + 1), 1)
knn_lane_kernel(const KnnArgs a0, const KnnArgs a1, int B0, int upb) {
    static_assert(ORDERED || !BQ, "Ball Query is fused into the ordered kernel only");
    constexpr int GQ = 32 * KL_QL;  // queries per group (warp)
    // cooked-tile swizzle bits and steps per hot-loop iteration: 3 and 8 for
    // one query per lane, 2 and 4 for two (registers)
    constexpr int KL_SB = KL_QL == 1 ? 3 : 2;
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool second = int(blockIdx.y) >= B0;
    const KnnArgs a = second ? a1 : a0;
    const int b = second ? int(blockIdx.y) - B0 : int(blockIdx.y);
    const int k = a.k;
    const float inf = __int_as_float(0x7f800000);

    StreamRing ring;
    int *flags = stream_carve(smem, ring);
    int *s_err = flags;
    unsigned long long *hk_all =
        reinterpret_cast<unsigned long long *>(smem + stream_smem_bytes());
    // BQ: per query slot its Ball Query state (hits, largest kept j, its
    // slot), after the heaps
    int4 *bq_st = reinterpret_cast<int4 *>(
        smem + stream_smem_bytes() +
        size_t(blockDim.x / 32 - 1) * 32 * KL_QL * size_t(k) * 8);

    const float *cref = ORDERED ? a.sref + size_t(b) * size_t(a.N) * 4
                                : a.ref + size_t(b) * size_t(a.N) * 3;
    const int Nb = valid_len(a.r_len, b, a.N);
    const int Qb = valid_len(a.q_len, b, a.Q);
    const int ntiles = (Nb + ST_T - 1) / ST_T;
    const int tstride = scramble_stride(ntiles);
    // ORDERED: part blockIdx.z of gridDim.z visits steps [it0, it1) of the
    // cloud's visiting order
    const int part = ORDERED ? static_cast<int>(blockIdx.z) : 0;
    const int nparts = ORDERED ? static_cast<int>(gridDim.z) : 1;
    const int it0 = static_cast<int>((static_cast<long long>(ntiles) * part) / nparts);
    const int nsteps_part =
        static_cast<int>((static_cast<long long>(ntiles) * (part + 1)) / nparts) - it0;
    const int nwarps = static_cast<int>(blockDim.x >> 5) - 1;  // consumers
    const int nbx = static_cast<int>(gridDim.x);
    const int bx = static_cast<int>(blockIdx.x);
    // ORDERED: the block's units [u0, u1) of the valid queries; else this
    // warp's group, strided over the cloud.  The warps that hold a valid
    // query (a prefix of the block's warps) consume the stream.
    const int u0 = ORDERED ? bx * upb : 0;
    const int u1 = ORDERED ? min(u0 + upb, (Qb + 31) / 32) : 0;
    const int g = warp * nbx + bx;
    const int gvalid = (Qb + GQ - 1) / GQ;
    const int nact = ORDERED ? max(0, min(nwarps, (u1 - u0 + KL_QL - 1) / KL_QL))
                             : (bx < gvalid ? min(nwarps, (gvalid - bx + nbx - 1) / nbx) : 0);
    if (ORDERED) {
        // rows past the cloud's valid length: padding, spread over the blocks
        if (warp == 0 && part == 0)
            for (int r = Qb + bx; r < a.Q; r += nbx)
                for (int e = lane; e < k; e += 32) {
                    a.out_idx[(size_t(b) * a.Q + r) * k + e] = -1;
                    a.out_dist[(size_t(b) * a.Q + r) * k + e] = 0.0f;
                }
        if (warp < nwarps && warp >= nact) return;
    } else if (warp < nwarps && warp >= nact) {
        // a group past the cloud's valid length: padding rows only
        const int r0 = min(a.Q, g * GQ), r1 = min(a.Q, r0 + GQ);
        const size_t e0 = (size_t(b) * a.Q + r0) * k;
        const size_t e1 = (size_t(b) * a.Q + r1) * k;
        for (size_t e = e0 + lane; e < e1; e += 32) {
            a.out_idx[e] = -1;
            a.out_dist[e] = 0.0f;
        }
        return;
    }
    if (nact == 0) return;  // the producer of a block without consumers
    if (threadIdx.x == 0) {
        stream_init(ring, nact);
        *s_err = 0;
    }
    // the filter's centre from up to 256 points spread over the cloud in
    // input order (the first points of a spatially sorted cloud would all
    // sit in one corner)
    const int fstep = max(1, Nb / ST_T);
    const FilterFrame fr = filter_frame(a.ref + size_t(b) * size_t(a.N) * 3,
                                        min(ST_T, Nb), 3 * fstep);
    // ORDERED: the home tile, where the middle query of the block's region
    // would sit among the references
    int home = 0;
    if (ORDERED && ntiles > 0) {
        const int pm = min(Qb - 1, u0 * 32 + (u1 - u0) * 16);
        const float *qm = a.squery + (size_t(b) * a.Q + pm) * 4;
        const unsigned code = mc_code(a.cframe + size_t(b) * 8, qm[0], qm[1], qm[2]);
        home = min(ntiles - 1, a.cstart[size_t(b) * (MC_CELLS + 1) + code] / ST_T);
    }
    // consumers and the producer only (the other warps have left)
    named_barrier_sync(1, unsigned(32 * (nact + 1)));
    // tile visited at step `it`: ORDERED outwards from home, else scrambled
    auto tile_at = [&](int itp) {
        const int it = it0 + itp;
        if (ORDERED) {
            const int off = (it & 1) ? (it + 1) >> 1 : -(it >> 1);
            int t = (home + off) % ntiles;
            return t < 0 ? t + ntiles : t;
        }
        return knn_tile_at(it, tstride, ntiles);
    };

    if (warp == nwarps) {  // producer warp
        const bool withhold = (a.stall & PC_STALL_TILE_STREAM) && blockIdx.x == 0 &&
                              blockIdx.y == 0 && blockIdx.z == 0;
        stream_produce<KL_SB, ORDERED>(ring, cref, Nb, nsteps_part, tile_at, fr, s_err,
                                       s_err, a.timeout_ns, withhold);
        return;
    }

    // query q of this lane: unit u0 + warp * KL_QL + q (ORDERED) or
    // g * KL_QL + q, query 32 * unit + lane; its heap is at slot
    // (warp * KL_QL + q) * 32 + lane, entries 32 apart.  The position (and
    // the output row) is recomputed at the end, not kept live through the
    // tile loop.
    auto query_pos = [&](int q) {
        const int unit = ORDERED ? u0 + warp * KL_QL + q : g * KL_QL + q;
        return unit * 32 + lane;
    };
    int qi[KL_QL];
    bool valid[KL_QL];
    float qx[KL_QL], qy[KL_QL], qz[KL_QL], qq[KL_QL], thr[KL_QL];
    float thr0[KL_QL];  // threshold of the seed bound (below)
    int seed_t[KL_QL];  // ORDERED: the seeded tile (-1: none), skipped here
    unsigned long long tk[KL_QL];  // heap root: the k-th best so far
    float2 ax[KL_QL], ay[KL_QL], az[KL_QL];
#pragma unroll
    for (int q = 0; q < KL_QL; ++q) {
        qi[q] = query_pos(q);
        valid[q] = qi[q] < Qb && (!ORDERED || (qi[q] >> 5) < u1);
        qx[q] = qy[q] = qz[q] = 0.f;
        if (valid[q]) {
            if (ORDERED) {
                const float4 p = reinterpret_cast<const float4 *>(
                    a.squery)[size_t(b) * a.Q + qi[q]];
                qx[q] = p.x;
                qy[q] = p.y;
                qz[q] = p.z;
            } else {
                const float *p = a.query + (size_t(b) * a.Q + qi[q]) * 3;
                qx[q] = p[0];
                qy[q] = p[1];
                qz[q] = p[2];
            }
        }
        const float xp = __fsub_rn(qx[q], fr.cx), yp = __fsub_rn(qy[q], fr.cy),
                    zp = __fsub_rn(qz[q], fr.cz);
        float axs, ays, azs;
        qq[q] = filter_query(xp, yp, zp, axs, ays, azs);
        ax[q] = make_float2(axs, axs);
        ay[q] = make_float2(ays, ays);
        az[q] = make_float2(azs, azs);
        tk[q] = KEY_EMPTY;
        unsigned long long *hk = hk_all + size_t(warp * KL_QL + q) * 32 * k + lane;
        for (int e = 0; e < k; ++e) hk[e * 32] = KEY_EMPTY;
        // ORDERED: the query's seeded tile was searched exactly by
        // knn_seed_kernel; part 0 starts from that heap, and every part skips
        // that tile.  The seed heap's root bounds the k-th smallest s32
        // (the s32 of the k-th of k distinct references), so until a part's
        // own heap is full its filter threshold is that bound instead of
        // +inf; afterwards the smaller of the two.
        float tau0 = inf;
        seed_t[q] = -1;
        if (ORDERED && valid[q]) {
            seed_t[q] = seed_tile(a, b, qi[q], qx[q], qy[q], qz[q], ntiles);
            const unsigned long long *sk = a.seed + (size_t(b) * a.Q + qi[q]) * k;
            const unsigned long long root = sk[0];
            if (key_j(root) != INT_MAX) tau0 = key_s(root);
            if (part == 0) {
                for (int e = 0; e < k; ++e) hk[e * 32] = sk[e];
                tk[q] = root;
            }
        }
        thr0[q] = valid[q] ? filter_threshold(tau0, qq[q]) : -inf;
        thr[q] = thr0[q];
        if constexpr (BQ) {
            if (valid[q]) {
                bq_st[(warp * KL_QL + q) * 32 + lane] = a.bq_state[size_t(b) * a.Q + qi[q]];
                thr[q] = fmaxf(thr0[q], filter_threshold(a.bq_R2, qq[q]));
            }
        }
    }

    // The tile loop for the first NQ query slots of each lane; returns true
    // when a wait for a stage ran out.  ORDERED with two slots, a warp left
    // with one unit (its second slot holds no valid query) runs it for one
    // slot: pass 1 at about half the cost, and half the live state.
    auto tile_loop = [&](auto nq_c) -> bool {
        constexpr int NQ = decltype(nq_c)::value;
        for (int it = 0; it < nsteps_part; ++it) {
            const int st = it % ST_STAGES;
            const WaitResult w = warp_wait(&ring.ready[st], unsigned((it / ST_STAGES) & 1),
                                           s_err, a.timeout_ns);
            if (w != WAIT_OK) return true;
            const float4 *ck = ring.cooked_tile(st);
            const int j0 = tile_at(it) * ST_T;
            const int cnt = min(ST_T, Nb - j0);
            const float4 *raw = ring.raw_copy(st);
            // whole rows of 8 steps (64 points); the cooked tile is padded to
            // ST_T points with points that pass only an infinite threshold
            const int nsteps = ((cnt + 63) >> 6) << 3;
            // pass 1: filter the whole tile, remembering which 8-point steps
            // let something through for which query (32 steps per tile)
            unsigned pend[KL_QL];
#pragma unroll
            for (int q = 0; q < KL_QL; ++q) pend[q] = 0;
            lane_pass1<NQ, KL_QL, KL_SB>(ck, nsteps, ax, ay, az, thr, pend);
            // ORDERED: a query's seeded tile is already in its heap (part 0)
            if (ORDERED) {
                const int tcur = j0 / ST_T;
#pragma unroll
                for (int q = 0; q < NQ; ++q)
                    if (tcur == seed_t[q]) pend[q] = 0;
            }
            // pass 2: the lanes with pending steps process them together (one
            // step per lane per round), exact s32 and heap insertion;
            // thresholds only tighten, so re-filtering with the current one is
            // still safe
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                if (!valid[q]) pend[q] = 0;
                unsigned long long *hk = hk_all + size_t(warp * KL_QL + q) * 32 * k + lane;
                while (__any_sync(FULL, pend[q] != 0)) {
                    if (pend[q] == 0) continue;
                    const int p = 4 * (__ffs(pend[q]) - 1);
                    pend[q] &= pend[q] - 1;
                    unsigned m = stream_mask<KL_SB, 4>(ck, p, ax[q], ay[q], az[q], thr[q]);
                    while (m) {
                        const int i = 2 * p + __ffs(m) - 1;
                        m &= m - 1;
                        if (i >= cnt) continue;
                        const float4 P = raw[raw_slot(i)];
                        const float sv = sqdist(qx[q], qy[q], qz[q], P.x, P.y, P.z);
                        // s32 >= +0; a NaN s32 has a key above KEY_EMPTY and
                        // is never accepted
                        const unsigned long long key =
                            sj_key(sv, ORDERED ? __float_as_int(P.w) : j0 + i);
                        if (key < tk[q]) {
                            tk[q] = heap_sift(hk, k, 0, key);
                            if (key_j(tk[q]) != INT_MAX) {
                                thr[q] = fminf(thr0[q],
                                               filter_threshold(key_s(tk[q]), qq[q]));
                                if constexpr (BQ)
                                    thr[q] = fmaxf(thr[q], filter_threshold(a.bq_R2, qq[q]));
                            }
                        }
                        if constexpr (BQ) {
                            if (sv < a.bq_R2) {
                                int4 &st = bq_st[(warp * KL_QL + q) * 32 + lane];
                                int hits = st.x, maxj = st.y, maxpos = st.z;
                                bq_keep(a.bq_rows + (size_t(b) * a.Q + query_pos(q)) * a.bq_K,
                                        a.bq_K, hits, maxj, maxpos, __float_as_int(P.w), sv);
                                st = make_int4(hits, maxj, maxpos, 0);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ring.empty[st]);  // tile no longer read
        }
        return false;
    };
    bool failed;
    if constexpr (ORDERED && KL_QL == 2) {
        if (u0 + warp * KL_QL + 1 >= u1)
            failed = tile_loop(std::integral_constant<int, 1>{});
        else
            failed = tile_loop(std::integral_constant<int, 2>{});
    } else {
        failed = tile_loop(std::integral_constant<int, KL_QL>{});
    }

    if (failed) {
        if (lane == 0) *s_err = 1;
        raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
    }
#pragma unroll
    for (int q = 0; q < KL_QL; ++q) {
        const int qp = query_pos(q);
        if (qp >= a.Q || (ORDERED && !valid[q])) continue;
        // output row: ORDERED, the query's original index
        const float4 *sq = reinterpret_cast<const float4 *>(a.squery);
        const int orow = ORDERED ? __float_as_int(sq[size_t(b) * a.Q + qp].w) : qp;
        const size_t row = size_t(b) * a.Q + orow;
        if constexpr (BQ) {  // the state for knn_bq_finish_kernel
            int4 st = bq_st[(warp * KL_QL + q) * 32 + lane];
            if (failed) st.x = -1;
            a.bq_state[size_t(b) * a.Q + qp] = st;
        }
        if (failed) {
            if (ORDERED && nparts > 1) {
                unsigned long long *pk =
                    a.part_keys + ((size_t(part) * gridDim.y + b) * a.Q + orow) * k;
                for (int e = 0; e < k; ++e) pk[e] = KEY_FAILED;
            } else {
                for (int e = 0; e < k; ++e) a.out_idx[row * k + e] = -1;
            }
            continue;
        }
        unsigned long long *hk = hk_all + size_t(warp * KL_QL + q) * 32 * k + lane;
        // heap sort: the largest entry moves to the end, k - 1 times
        for (int n = k - 1; n > 0; --n) {
            const unsigned long long key = hk[n * 32];
            hk[n * 32] = hk[0];
            heap_sift(hk, n, 0, key);
        }
        if (ORDERED && nparts > 1) {  // this part's sorted keys, merged later
            unsigned long long *pk =
                a.part_keys + ((size_t(part) * gridDim.y + b) * a.Q + orow) * k;
            for (int e = 0; e < k; ++e) pk[e] = hk[e * 32];
            continue;
        }
        const int kv = valid[q] ? min(k, Nb) : 0;
        for (int e = 0; e < k; ++e) {
            const unsigned long long key = hk[e * 32];
            const float sv = key_s(key);
            a.out_idx[row * k + e] = e < kv ? int64_t(key_j(key)) : int64_t(-1);
            a.out_dist[row * k + e] = e < kv ? (a.squared ? sv : __fsqrt_rn(sv)) : 0.0f;
        }
    }
}

// The k smallest keys of a valid query row over the parts' sorted lists
// (ORDERED with the references split): one thread per row.
__global__ void __launch_bounds__(256) knn_merge_parts_kernel(const KnnArgs a, int B,
                                                              int nparts) {
    const int b = blockIdx.y;
    const int r = blockIdx.x * 256 + threadIdx.x;
    if (r >= valid_len(a.q_len, b, a.Q)) return;
    const int k = a.k;
    const int kv = min(k, valid_len(a.r_len, b, a.N));
    const size_t stride = size_t(B) * a.Q * k;  // between parts
    const unsigned long long *pk = a.part_keys + (size_t(b) * a.Q + r) * k;
    int ptr[8];
    for (int p = 0; p < nparts; ++p) ptr[p] = 0;
    const size_t row = size_t(b) * a.Q + r;
    for (int p = 0; p < nparts; ++p)
        if (pk[p * stride] == KEY_FAILED) {  // a part stopped: unfinished row
            for (int e = 0; e < k; ++e) {
                a.out_idx[row * k + e] = -1;
                a.out_dist[row * k + e] = 0.0f;
            }
            return;
        }
    for (int e = 0; e < k; ++e) {
        unsigned long long best = KEY_EMPTY;
        int bp = -1;
        for (int p = 0; p < nparts; ++p)
            if (ptr[p] < k) {
                const unsigned long long key = pk[p * stride + ptr[p]];
                if (key < best) {
                    best = key;
                    bp = p;
                }
            }
        if (bp >= 0) ++ptr[bp];
        const float sv = key_s(best);
        a.out_idx[row * k + e] = e < kv ? int64_t(key_j(best)) : int64_t(-1);
        a.out_dist[row * k + e] = e < kv ? (a.squared ? sv : __fsqrt_rn(sv)) : 0.0f;
    }
}

// Ball Query fused into the ordered lane kNN: a query's kept hits (the bq_K
// smallest indices with s32 < R2, in no order) sorted by index into its
// output row, (-1, 0) in the slots after them; a query whose search stopped
// on a timeout gets (-1, 0) throughout.  One warp per query (in the query
// order), at most 64 hits: a hit's place is the number of kept indices
// below its own (the indices are distinct).
constexpr int BQ_FUSE_MAX_K = 64;

__global__ void __launch_bounds__(256) knn_bq_finish_kernel(const KnnArgs a) {
    const int b = blockIdx.y;
    const int qp = blockIdx.x * 8 + static_cast<int>(threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (qp >= a.Q) return;
    const int K = a.bq_K;
    const size_t at = size_t(b) * a.Q + qp;
    const int4 st = a.bq_state[at];
    const int orow = __float_as_int(reinterpret_cast<const float4 *>(a.squery)[at].w);
    const size_t row = (size_t(b) * a.Q + orow) * K;
    const int cnt = st.x < 0 ? 0 : min(st.x, K);
    const int2 *src = a.bq_rows + at * K;
    const int2 e0 = lane < cnt ? src[lane] : make_int2(INT_MAX, 0);
    const int2 e1 = lane + 32 < cnt ? src[lane + 32] : make_int2(INT_MAX, 0);
    int r0 = 0, r1 = 0;
    for (int m = 0; m < cnt; ++m) {
        const int jm = __shfl_sync(FULL, m < 32 ? e0.x : e1.x, m & 31);
        r0 += jm < e0.x ? 1 : 0;
        r1 += jm < e1.x ? 1 : 0;
    }
    if (lane < cnt) {
        a.bq_out_idx[row + r0] = e0.x;
        a.bq_out_d2[row + r0] = __int_as_float(e0.y);
    }
    if (lane + 32 < cnt) {
        a.bq_out_idx[row + r1] = e1.x;
        a.bq_out_d2[row + r1] = __int_as_float(e1.y);
    }
    for (int e = cnt + lane; e < K; e += 32) {
        a.bq_out_idx[row + e] = -1;
        a.bq_out_d2[row + e] = 0.0f;
    }
}

template <int QL, bool ORDERED = false, bool BQ = false>
cudaError_t launch_knn_lane(const DeviceInfo &dev, const KnnArgs &a0, int64_t B0,
                            const KnnArgs &a1, int64_t B1, cudaStream_t stream,
                            int nparts = 1) {
    const int64_t GQ = 32 * QL;
    const int64_t Q = std::max<int64_t>(a0.Q, B1 > 0 ? a1.Q : 0);
    const int64_t G = (Q + GQ - 1) / GQ;  // groups per cloud
    const int64_t total = G * (B0 + B1) * nparts;
    if (total == 0) return cudaSuccess;
    const int64_t nsm = std::max(1, dev.sm_count - sm_reserve());
    // consumer warps per block: shared memory bounds it too (k * 8 bytes per
    // query, and 16 for the fused Ball Query's state); a block per SM and wave
    const int64_t per_warp = GQ * (int64_t(a0.k) * 8 + (BQ ? 16 : 0));
    const int64_t wmax = std::max<int64_t>(
        1, std::min<int64_t>(kl_wmax(QL), (int64_t(dev.smem_per_block_optin) -
                                       int64_t(stream_smem_bytes())) / per_warp));
    int64_t W, nbx, upb = 0;
    if (ORDERED) {
        // units of 32 queries: a block takes upb consecutive units, about the
        // same number per SM (to half a warp with two slots per lane)
        const int64_t U = (Q + 31) / 32;  // units per cloud
        const int64_t utotal = U * (B0 + B1) * nparts;
        const int64_t umax = wmax * QL;
        const int64_t waves = (utotal + nsm * umax - 1) / (nsm * umax);
        upb = std::min(std::min(umax, U), (utotal + nsm * waves - 1) / (nsm * waves));
        W = (upb + QL - 1) / QL;
        nbx = (U + upb - 1) / upb;
    } else {
        const int64_t waves = (total + nsm * wmax - 1) / (nsm * wmax);
        W = std::min(std::min(wmax, G), (total + nsm * waves - 1) / (nsm * waves));
        nbx = (G + W - 1) / W;
    }
    const size_t smem = knn_lane_smem(a0.k, QL, int(W)) + (BQ ? size_t(W) * GQ * 16 : 0);
    cudaError_t e = cudaFuncSetAttribute(
        knn_lane_kernel<QL, ORDERED, BQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(nbx), static_cast<unsigned>(B0 + B1),
              static_cast<unsigned>(nparts));
    knn_lane_kernel<QL, ORDERED, BQ>
        <<<grid, unsigned(32 * (W + 1)), smem, stream>>>(a0, a1, int(B0), int(upb));
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The spatial order of the ORDERED lane kernel, per cloud:
//   1. frame: bounding box of (up to) 4096 valid references spread evenly
//      over the cloud (whatever its storage order), and 2^MC_BITS cells per
//      axis over it;
//   2. count the valid references per cell code; exclusive scan;
//   3. scatter them as (x, y, z, original index) in code order (the order
//      within a cell is whatever the atomics give: the kNN result does not
//      depend on it); the same for the valid queries, with the references'
//      frame, unless the query set is the reference set.
// ---------------------------------------------------------------------------
constexpr int MC_SAMPLE = 4096;

__global__ void __launch_bounds__(256) mc_frame_kernel(const float *pts,
                                                       const int64_t *lens, int n,
                                                       float *frame) {
    __shared__ float red[6][8];
    const int b = blockIdx.x;
    const int nv = valid_len(lens, b, n);
    const int step = max(1, nv / MC_SAMPLE);
    const int nb = min(nv, MC_SAMPLE);
    const float *c = pts + size_t(b) * n * 3;
    const float inf = __int_as_float(0x7f800000);
    float lo[3] = {inf, inf, inf}, hi[3] = {-inf, -inf, -inf};
    for (int i = threadIdx.x; i < nb; i += 256)
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const float v = c[size_t(i) * step * 3 + d];
            lo[d] = fminf(lo[d], v);
            hi[d] = fmaxf(hi[d], v);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            lo[d] = fminf(lo[d], __shfl_xor_sync(FULL, lo[d], o));
            hi[d] = fmaxf(hi[d], __shfl_xor_sync(FULL, hi[d], o));
        }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            red[d][w] = lo[d];
            red[3 + d][w] = hi[d];
        }
    __syncthreads();
    if (threadIdx.x < 3) {
        const int d = threadIdx.x;
        float l = inf, h = -inf;
        for (int i = 0; i < 8; ++i) {
            l = fminf(l, red[d][i]);
            h = fmaxf(h, red[3 + d][i]);
        }
        const float ext = h - l;
        const bool ok = ext > 0.0f && ext < 3e38f && l > -3e38f;
        frame[size_t(b) * 8 + d] = ok ? l : 0.0f;
        frame[size_t(b) * 8 + 3 + d] = ok ? float(1 << MC_BITS) / ext : 0.0f;
    }
}

__global__ void __launch_bounds__(256) mc_count_kernel(const float *pts,
                                                       const int64_t *lens, int n,
                                                       const float *frame, int *hist) {
    const int b = blockIdx.y;
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= valid_len(lens, b, n)) return;
    const float *p = pts + (size_t(b) * n + i) * 3;
    const unsigned code = mc_code(frame + size_t(b) * 8, p[0], p[1], p[2]);
    atomicAdd(&hist[size_t(b) * (MC_CELLS + 1) + code], 1);
}

// Exclusive scan of each cloud's MC_CELLS counts into start[0 .. MC_CELLS]
// (start[MC_CELLS] = total) and cursor (a copy of the starts), in chunks of
// 1024 counts, one block each: mc_chunk_sum_kernel totals every chunk,
// mc_scan_kernel scans a chunk and adds the totals of the chunks before it.
constexpr int MC_CHUNKS = MC_CELLS / 1024;

// Inclusive scan of v over the 1024 threads of the block (wsum: 32 ints of
// shared memory); returns the block total in *total.
__device__ __forceinline__ int block_scan_1024(int v, int *wsum, int *total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        int z = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, z, o);
            if (lane >= o) z += y;
        }
        wsum[lane] = z;
    }
    __syncthreads();
    *total = wsum[31];
    return x + (w > 0 ? wsum[w - 1] : 0);
}

__global__ void __launch_bounds__(1024) mc_chunk_sum_kernel(const int *hist, int *chunk) {
    __shared__ int wsum[32];
    const int b = blockIdx.y, c = blockIdx.x;
    const int v = hist[size_t(b) * (MC_CELLS + 1) + c * 1024 + threadIdx.x];
    int total;
    block_scan_1024(v, wsum, &total);
    if (threadIdx.x == 0) chunk[b * MC_CHUNKS + c] = total;
}

__global__ void __launch_bounds__(1024) mc_scan_kernel(const int *hist, const int *chunk,
                                                       int *start, int *cursor) {
    __shared__ int wsum[32];
    const int b = blockIdx.y, c = blockIdx.x;
    int before = 0;  // the chunks before this one, in order
    for (int i = 0; i < c; ++i) before += chunk[b * MC_CHUNKS + i];
    const size_t e = size_t(b) * (MC_CELLS + 1) + c * 1024 + threadIdx.x;
    const int v = hist[e];
    int total;
    const int incl = block_scan_1024(v, wsum, &total);
    start[e] = before + incl - v;
    cursor[e] = before + incl - v;
    if (c == MC_CHUNKS - 1 && threadIdx.x == 1023)
        start[size_t(b) * (MC_CELLS + 1) + MC_CELLS] = before + total;
}

__global__ void __launch_bounds__(256) mc_scatter_kernel(const float *pts,
                                                         const int64_t *lens, int n,
                                                         const float *frame, int *cursor,
                                                         float4 *out) {
    const int b = blockIdx.y;
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= valid_len(lens, b, n)) return;
    const float *p = pts + (size_t(b) * n + i) * 3;
    const float x = p[0], y = p[1], z = p[2];
    const unsigned code = mc_code(frame + size_t(b) * 8, x, y, z);
    const int pos = atomicAdd(&cursor[size_t(b) * (MC_CELLS + 1) + code], 1);
    out[size_t(b) * n + pos] = make_float4(x, y, z, __int_as_float(i));
}

// Parts of the ORDERED lane kNN: with few queries against many references
// the references are split into parts (blocks of the same queries, other
// tiles), about 10 warps per SM.
int ordered_nparts(const DeviceInfo &dev, int64_t B, int64_t Q, int64_t N, int QL) {
    const int64_t groups = B * ((Q + 32 * QL - 1) / (32 * QL));
    const int64_t ntiles = (N + ST_T - 1) / ST_T;
    const int64_t want =
        (int64_t(std::max(1, dev.sm_count - sm_reserve())) * 10 + groups - 1) / groups;
    return int(std::max<int64_t>(1, std::min<int64_t>({8, want, ntiles / 8})));
}

// Ball Query fused into the ORDERED lane kNN (one part, K <= 64).
struct BqFuse {
    float R2;
    int K;
    float *out_d2;
    int64_t *out_idx;
};

// The ORDERED lane kNN: order the clouds, then one lane-kernel launch over
// `nparts` parts of the references (ordered_nparts; one with `fuse`, which
// adds the Ball Query of the same queries to the same launch).  The scratch
// memory is stream-ordered (allocated and freed on `stream`).
template <int QL>
cudaError_t launch_knn_ordered(const DeviceInfo &dev, KnnArgs a, int64_t B, int nparts,
                               cudaStream_t stream, const BqFuse *fuse = nullptr) {
    const bool self = a.query == a.ref && a.Q == a.N && a.q_len == a.r_len;
    const size_t cells = size_t(B) * (MC_CELLS + 1) * sizeof(int);
    const size_t off_frame = 0;
    // hist_r then hist_q (zeroed together)
    const size_t off_hist = (size_t(B) * 8 * sizeof(float) + 255) & ~size_t(255);
    const size_t off_start = off_hist + 2 * cells;
    const size_t off_cur = off_start + cells;
    const size_t off_curq = off_cur + cells;
    const size_t off_chunk = (off_curq + cells + 255) & ~size_t(255);
    const size_t off_sref =
        (off_chunk + 2 * size_t(B) * MC_CHUNKS * sizeof(int) + 255) & ~size_t(255);
    const size_t off_sq = off_sref + ((size_t(B) * a.N * 16 + 255) & ~size_t(255));
    if (fuse && (nparts != 1 || fuse->K > BQ_FUSE_MAX_K)) return cudaErrorInvalidValue;
    const size_t off_pk = off_sq + ((self ? 0 : size_t(B) * a.Q * 16 + 255) & ~size_t(255));
    const size_t off_seed =
        off_pk + ((nparts > 1 ? size_t(nparts) * B * a.Q * size_t(a.k) * 8 : 0) + 255 &
                  ~size_t(255));
    // the fused Ball Query: kept hits [B][Q][K] (8 bytes each), state [B][Q]
    const size_t off_bq_rows =
        (off_seed + size_t(B) * a.Q * size_t(a.k) * 8 + 255) & ~size_t(255);
    const size_t off_bq_state =
        off_bq_rows + ((fuse ? size_t(B) * a.Q * size_t(fuse->K) * 8 : 0) + 255 & ~size_t(255));
    const size_t total = off_bq_state + (fuse ? size_t(B) * a.Q * 16 : 0);
    char *base = nullptr;
    cudaError_t e = scratch_alloc(dev, reinterpret_cast<void **>(&base), total, stream);
    if (e != cudaSuccess) return e;
    float *frame = reinterpret_cast<float *>(base + off_frame);
    int *hist = reinterpret_cast<int *>(base + off_hist);
    int *start = reinterpret_cast<int *>(base + off_start);
    int *cur = reinterpret_cast<int *>(base + off_cur);
    int *curq = reinterpret_cast<int *>(base + off_curq);
    int *chunk = reinterpret_cast<int *>(base + off_chunk);
    int *chunkq = chunk + B * MC_CHUNKS;
    float4 *sref = reinterpret_cast<float4 *>(base + off_sref);
    float4 *sq = self ? sref : reinterpret_cast<float4 *>(base + off_sq);
    int *histq = hist + size_t(B) * (MC_CELLS + 1);
    e = cudaMemsetAsync(hist, 0, 2 * cells, stream);
    const dim3 gr(unsigned((a.N + 255) / 256), unsigned(B));
    const dim3 gq(unsigned((a.Q + 255) / 256), unsigned(B));
    if (e == cudaSuccess) {
        mc_frame_kernel<<<unsigned(B), 256, 0, stream>>>(a.ref, a.r_len, a.N, frame);
        mc_count_kernel<<<gr, 256, 0, stream>>>(a.ref, a.r_len, a.N, frame, hist);
        const dim3 gc(MC_CHUNKS, unsigned(B));
        mc_chunk_sum_kernel<<<gc, 1024, 0, stream>>>(hist, chunk);
        mc_scan_kernel<<<gc, 1024, 0, stream>>>(hist, chunk, start, cur);
        mc_scatter_kernel<<<gr, 256, 0, stream>>>(a.ref, a.r_len, a.N, frame, cur, sref);
        if (!self) {
            // the query starts are only cursors: scan into curq twice over
            mc_count_kernel<<<gq, 256, 0, stream>>>(a.query, a.q_len, a.Q, frame, histq);
            mc_chunk_sum_kernel<<<gc, 1024, 0, stream>>>(histq, chunkq);
            mc_scan_kernel<<<gc, 1024, 0, stream>>>(histq, chunkq, curq, curq);
            mc_scatter_kernel<<<gq, 256, 0, stream>>>(a.query, a.q_len, a.Q, frame, curq,
                                                      sq);
        }
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) {
        a.sref = reinterpret_cast<const float *>(sref);
        a.squery = reinterpret_cast<const float *>(sq);
        a.cstart = start;
        a.cframe = frame;
        a.part_keys =
            nparts > 1 ? reinterpret_cast<unsigned long long *>(base + off_pk) : nullptr;
        unsigned long long *seed = reinterpret_cast<unsigned long long *>(base + off_seed);
        a.seed = seed;
        if (fuse) {
            a.bq_rows = reinterpret_cast<int2 *>(base + off_bq_rows);
            a.bq_state = reinterpret_cast<int4 *>(base + off_bq_state);
            a.bq_R2 = fuse->R2;
            a.bq_K = fuse->K;
            a.bq_out_d2 = fuse->out_d2;
            a.bq_out_idx = fuse->out_idx;
        }
        const size_t seed_smem = size_t(SEED_THREADS) * size_t(a.k) * 8;
        e = cudaFuncSetAttribute(knn_seed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(seed_smem));
        if (e == cudaSuccess) {
            knn_seed_kernel<<<dim3(unsigned((a.Q + SEED_THREADS - 1) / SEED_THREADS),
                                   unsigned(B)),
                              SEED_THREADS, seed_smem, stream>>>(a, seed);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess)
            e = fuse ? launch_knn_lane<QL, true, true>(dev, a, B, a, 0, stream, 1)
                     : launch_knn_lane<QL, true>(dev, a, B, a, 0, stream, nparts);
        if (e == cudaSuccess && fuse) {
            knn_bq_finish_kernel<<<dim3(unsigned((a.Q + 7) / 8), unsigned(B)), 256, 0,
                                   stream>>>(a);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess && nparts > 1) {
            const dim3 gm(unsigned((a.Q + 255) / 256), unsigned(B));
            knn_merge_parts_kernel<<<gm, 256, 0, stream>>>(a, int(B), nparts);
            e = cudaGetLastError();
        }
    }
    const cudaError_t f = scratch_free(base, stream);
    return e != cudaSuccess ? e : f;
}

template <int KPL>
cudaError_t launch_knn_t(const DeviceInfo &dev, const KnnArgs &a0, int64_t B,
                         int64_t Q, cudaStream_t stream) {
    KnnArgs a = a0;
    const size_t per_q = knn_per_query_smem(a.k);
    const int slots = dev.sm_count * 2;
    // queries per warp: spread B*Q over about one wave of 2 blocks per SM
    const int64_t bpc_target = std::max<int64_t>(1, slots / std::max<int64_t>(B, 1));
    int64_t G = (Q + KNN_CWARPS * bpc_target - 1) / (KNN_CWARPS * bpc_target);
    const size_t budget =
        std::min<size_t>(dev.smem_per_block_optin, dev.smem_per_sm / 2 - 2048);
    const int64_t gmax = std::max<int64_t>(
        1, int64_t((budget - knn_fixed_smem()) / (KNN_CWARPS * per_q)));
    G = std::max<int64_t>(1, std::min(G, gmax));
    a.q_per_warp = static_cast<int>(G);
    const int64_t bpc = (Q + KNN_CWARPS * G - 1) / (KNN_CWARPS * G);
    const size_t smem = knn_fixed_smem() + size_t(KNN_CWARPS) * G * per_q;
    cudaError_t e = cudaFuncSetAttribute(
        knn_kernel<KPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(bpc), static_cast<unsigned>(B));
    knn_kernel<KPL><<<grid, KNN_THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

namespace {

KnnArgs make_knn_args(const DeviceInfo &dev, const float *query, int64_t Q,
                      const float *ref, int64_t N, int k, const int64_t *q_len,
                      const int64_t *r_len, bool squared, float *out_dist,
                      int64_t *out_idx) {
    KnnArgs a{};
    a.query = query;
    a.ref = ref;
    a.q_len = q_len;
    a.r_len = r_len;
    a.Q = static_cast<int>(Q);
    a.N = static_cast<int>(N);
    a.k = k;
    a.squared = squared ? 1 : 0;
    a.out_dist = out_dist;
    a.out_idx = out_idx;
    a.status = dev.status_word;
    a.timeout_ns = wait_timeout_ns();
    a.stall = debug_stall();
    return a;
}

}  // namespace

cudaError_t launch_knn_pair(const DeviceInfo &dev, int64_t B, int k, bool squared,
                            const float *q0, int64_t Q0, const float *r0, int64_t N0,
                            const int64_t *ql0, const int64_t *rl0, float *d0,
                            int64_t *i0, const float *q1, int64_t Q1,
                            const float *r1, int64_t N1, const int64_t *ql1,
                            const int64_t *rl1, float *d1, int64_t *i1,
                            cudaStream_t stream) {
    if (k > 32 || B * 2 > 65535) {
        cudaError_t e = launch_knn(dev, q0, B, Q0, r0, N0, k, ql0, rl0, squared, d0,
                                   i0, stream);
        if (e != cudaSuccess) return e;
        return launch_knn(dev, q1, B, Q1, r1, N1, k, ql1, rl1, squared, d1, i1,
                          stream);
    }
    const KnnArgs a0 = make_knn_args(dev, q0, Q0, r0, N0, k, ql0, rl0, squared, d0, i0);
    const KnnArgs a1 = make_knn_args(dev, q1, Q1, r1, N1, k, ql1, rl1, squared, d1, i1);
    if (k <= 16) return launch_knn_lane<2>(dev, a0, B, a1, B, stream);
    return launch_knn_lane<1>(dev, a0, B, a1, B, stream);
}

cudaError_t launch_knn(const DeviceInfo &dev, const float *query, int64_t B,
                       int64_t Q, const float *ref, int64_t N, int k,
                       const int64_t *q_len, const int64_t *r_len, bool squared,
                       float *out_dist, int64_t *out_idx,
                       cudaStream_t stream) {
    const KnnArgs a = make_knn_args(dev, query, Q, ref, N, k, q_len, r_len, squared,
                                    out_dist, out_idx);
    // large clouds with k >= 2: the spatial order (a few extra launches)
    // pays for itself many times over in candidate insertions
    const bool ordered = k >= 2 && k <= 32 && N >= 16384 && Q >= 4096 && B <= 64;
    // few query groups (under a quarter of the SMs would hold a warp): one
    // warp per query with the warp-list kernel keeps every SM busy (GB300,
    // 64 queries vs 1024 points, k = 16: 0.045 ms vs 0.21 ms with the lane
    // kernel's single warp)
    if (B * ((Q + 31) / 32) * 4 < dev.sm_count) {
        if (k <= 64) return launch_knn_t<2>(dev, a, B, Q, stream);
        if (k <= 128) return launch_knn_t<4>(dev, a, B, Q, stream);
        return launch_knn_t<8>(dev, a, B, Q, stream);
    }
    if (ordered && k <= 16)
        return launch_knn_ordered<2>(dev, a, B, ordered_nparts(dev, B, Q, N, 2), stream);
    if (ordered)
        return launch_knn_ordered<1>(dev, a, B, ordered_nparts(dev, B, Q, N, 1), stream);
    if (k <= 16) return launch_knn_lane<2>(dev, a, B, a, 0, stream);
    if (k <= 32) return launch_knn_lane<1>(dev, a, B, a, 0, stream);
    if (k <= 64) return launch_knn_t<2>(dev, a, B, Q, stream);
    if (k <= 128) return launch_knn_t<4>(dev, a, B, Q, stream);
    return launch_knn_t<8>(dev, a, B, Q, stream);
}

namespace {
// The fused pass's conditions, given the ordered kNN's part count.
bool fused_applies(int64_t B, int64_t Q, int64_t N, int k, float r32, int64_t K,
                   int nparts) {
    const float R2 = r32 * r32;
    return k >= 2 && k <= 32 && N >= 16384 && Q >= 4096 && B <= 64 &&
           K <= BQ_FUSE_MAX_K && R2 > 0.0f && R2 <= 3e38f && nparts == 1;
}
}  // namespace

bool knn_ball_query_fused(const DeviceInfo &dev, int64_t B, int64_t Q, int64_t N,
                          int k, float r32, int64_t K) {
    return fused_applies(B, Q, N, k, r32, K, ordered_nparts(dev, B, Q, N, k <= 16 ? 2 : 1));
}

cudaError_t launch_knn_ball_query(const DeviceInfo &dev, const float *query, int64_t B,
                                  int64_t Q, const float *ref, int64_t N, int k,
                                  float *knn_dist, int64_t *knn_idx, float r32, int64_t K,
                                  float *bq_dist2, int64_t *bq_idx, cudaStream_t stream) {
    const int nparts = ordered_nparts(dev, B, Q, N, k <= 16 ? 2 : 1);
    if (!fused_applies(B, Q, N, k, r32, K, nparts)) {
        const cudaError_t e = launch_knn(dev, query, B, Q, ref, N, k, nullptr, nullptr,
                                         false, knn_dist, knn_idx, stream);
        if (e != cudaSuccess) return e;
        return launch_ball_query(dev, query, B, Q, ref, N, nullptr, nullptr, r32, K,
                                 bq_dist2, bq_idx, stream);
    }
    const KnnArgs a = make_knn_args(dev, query, Q, ref, N, k, nullptr, nullptr, false,
                                    knn_dist, knn_idx);
    const BqFuse fuse{r32 * r32, int(K), bq_dist2, bq_idx};
    if (k <= 16) return launch_knn_ordered<2>(dev, a, B, nparts, stream, &fuse);
    return launch_knn_ordered<1>(dev, a, B, nparts, stream, &fuse);
}

}  // namespace pcn
