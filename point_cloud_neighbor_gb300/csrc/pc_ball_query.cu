// pc_ball_query.cu -- dense first-K Ball Query on sm_103a.
//
// Operator (mps-pointops project page, "Ball Query: first K within a
// radius"; "Numerical contracts", "Selection and output"): with
// R2 = fl32(fl32(r) * fl32(r)), reference j is accepted iff s < R2; the
// first K accepted indices in input order are returned with their squared
// distances, unused slots hold (-1, 0).
//
// Design (one launch, no scratch memory; with few queries against many
// references, the references split into parts plus a merge, see below):
//  * A block has BQ_CWARPS consumer warps and one producer warp.  Consumer
//    warp w owns G queries of one cloud, kept in shared memory as the filter
//    constants of pc_filter.cuh duplicated for the packed instructions,
//    (-2x', -2x', -2y', -2y') and (-2z', -2z', thr, query index), plus the
//    raw coordinates and the hit count.
//  * The producer's lane 0 streams reference tiles of BQ_T = 32 * BQ_R points
//    strictly in input order through a BQ_STAGES ring (TMA bulk copies,
//    full/empty mbarriers); consumer warps derive the centred coordinates
//    and w' of their points into registers (lane l holds tile points
//    l + 32 r, so for each r the warp holds 32 consecutive references in
//    lane order) and release the raw tile once their queries are done.
//  * Per (query, tile) each lane evaluates the conservative filter for its
//    BQ_R points (three packed FMAs per pair) and one vote asks whether any
//    may be inside the radius; the hot loop is only the FMAs, the compares
//    and the vote.  On a vote (rare) the slow path computes the exact s32
//    from the raw tile in shared memory and, per r, a ballot gives the hits
//    among 32 consecutive references and __popc(ballot & lanemask_lt) gives
//    each hit its rank, so a hit is written straight to slot (hits so far +
//    rank): input order is kept without any sort.
//  * A query stops at K hits: it is swapped behind the still-active queries
//    of its warp, so the hot loop tests nothing per query.  When every query
//    of a block is full, a stop flag ends the block: the producer stops
//    issuing tiles (after letting its copies in flight land) and the
//    consumers leave the tile loop.
#include "pointcloud.h"
#include "pc_device.cuh"
#include "pc_filter.cuh"
#include "pc_internal.h"
#include "pc_stream.cuh"
#include "pc_tiles.cuh"

#include <algorithm>

namespace pcn {
namespace {

constexpr int BQ_R = 8;  // reference points per lane per tile
constexpr int BQ_CWARPS = 8;
// references split into parts when a warp would hold fewer queries than this
constexpr int BQ_MIN_QUERIES_PER_WARP = 24;
constexpr int64_t BQ_MAX_PARTS = 8;
constexpr int BQ_THREADS = 32 * (BQ_CWARPS + 1);
constexpr unsigned FULL = 0xffffffffu;
static_assert(32 * BQ_R == ST_T, "a lane holds 8 of a stream tile's points");

struct BqArgs {
    const float *query;
    const float *ref;
    const int64_t *q_len;  // valid queries per cloud (NULL: Q)
    const int64_t *r_len;  // valid references per cloud (NULL: N)
    int Q, N;
    float R2;
    int K;
    int q_per_warp;
    float *out_dist2;
    int64_t *out_idx;
    int *status;
    uint64_t timeout_ns;
    int stall;  // PC_STALL_* testing flags
    // references split into gridDim.z parts (few queries against many
    // references): part p records its first K hits per row in
    // part_idx/part_d2 [p][B][Q][K] and their number in part_cnt [p][B][Q]
    // (-1: the part stopped on a timeout); bq_merge_parts_kernel joins them
    int64_t *part_idx;
    float *part_d2;
    int *part_cnt;
};

struct __align__(16) BqSlot {
    float4 axy;  // (-2x', -2x', -2y', -2y')   centred coordinates
    float4 azt;  // (-2z', -2z', thr, query index in warp (int bits))
    float4 raw;  // (x, y, z, hits so far (int bits))
};

// Swizzle bits of the prepared stages: lanes read pairs l + 32 r, i.e. four
// consecutive pairs of each of eight steps, and with 3 bits two consecutive
// steps use complementary halves of the bank groups.
constexpr int BQ_SB = 3;

__host__ __device__ constexpr size_t bq_fixed_smem() { return stream_smem_bytes(); }
// the query slots that follow hold float4s
static_assert(bq_fixed_smem() % alignof(BqSlot) == 0, "query slots 16-byte aligned");

// Valid length of cloud b: lens[b] clamped to [0, full], or full.
__device__ __forceinline__ int valid_len(const int64_t *lens, int b, int full) {
    if (lens == nullptr) return full;
    const int64_t v = lens[b];
    return v < 0 ? 0 : (v > full ? full : static_cast<int>(v));
}

// Slow path, taken only when a vote let a pair through.  Lane l holds the
// pairs l + 32 r (points 2 (l + 32 r) + h, bit 2r + h of its filter mask),
// so for each r the warp holds the 64 consecutive references
// [64 r, 64 r + 64) in (lane, h) order.  The mask is recomputed, points that
// pass get their exact s32 from the stage's raw copy, and hits are recorded
// in input order: two ballots (h = 0, 1) rank every hit of the row.
// Returns the new hit count (<= K).
__device__ __forceinline__ int bq_record(const float4 *raw,
                                         const float2 (&rx)[BQ_R / 2],
                                         const float2 (&ry)[BQ_R / 2],
                                         const float2 (&rz)[BQ_R / 2],
                                         const float2 (&rw)[BQ_R / 2],
                                         float4 axy, float4 azt, const float4 q,
                                         int hits, int j0, int cnt, float R2,
                                         int K, size_t row, float *out_dist2,
                                         int64_t *out_idx) {
    const int lane = static_cast<int>(lane_id());
    const unsigned pm = filter_mask8(rx, ry, rz, rw, axy, azt);
    // rows r where some lane may hold a hit, in increasing r (input order)
    const unsigned any = __reduce_or_sync(FULL, pm);
    unsigned rows = (any | (any >> 1)) & 0x55u;
    const unsigned lt = lanemask_lt();
    while (rows) {
        const int r = (__ffs(rows) - 1) >> 1;
        rows &= rows - 1;
        float s[2] = {0.f, 0.f};
        bool hit[2] = {false, false};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = 2 * (lane + 32 * r) + h;  // point in the tile
            if (((pm >> (2 * r + h)) & 1u) && i < cnt) {
                const float4 p = raw[raw_slot(i)];
                s[h] = sqdist(q.x, q.y, q.z, p.x, p.y, p.z);
                hit[h] = s[h] < R2;
            }
        }
        const unsigned b0 = __ballot_sync(FULL, hit[0]);
        const unsigned b1 = __ballot_sync(FULL, hit[1]);
        if (b0 | b1) {
            const int before = hits + __popc(b0 & lt) + __popc(b1 & lt);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pos = before + (h == 1 && hit[0] ? 1 : 0);
                if (hit[h] && pos < K) {
                    out_idx[row * K + pos] = j0 + 2 * (lane + 32 * r) + h;
                    out_dist2[row * K + pos] = s[h];
                }
            }
            hits += __popc(b0) + __popc(b1);
            if (hits >= K) break;
        }
    }
    return min(hits, K);
}

__global__ void __launch_bounds__(BQ_THREADS, 2) bq_kernel(const BqArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int G = a.q_per_warp;
    const int K = a.K;

    StreamRing ring;
    int *flags = stream_carve(smem, ring);
    int *s_err = flags;
    int *s_stop = flags + 1;
    int *s_ndone = flags + 2;
    BqSlot *slots_all = reinterpret_cast<BqSlot *>(smem + bq_fixed_smem());

    const float *cref = a.ref + size_t(b) * size_t(a.N) * 3;
    const int Nb = valid_len(a.r_len, b, a.N);
    const int Qb = valid_len(a.q_len, b, a.Q);
    const int ntiles_all = (Nb + ST_T - 1) / ST_T;
    // part blockIdx.z of gridDim.z: tiles [t0, t0 + ntiles) of the cloud
    const int part = static_cast<int>(blockIdx.z), nparts = static_cast<int>(gridDim.z);
    const int t0 = static_cast<int>((static_cast<long long>(ntiles_all) * part) / nparts);
    const int ntiles =
        static_cast<int>((static_cast<long long>(ntiles_all) * (part + 1)) / nparts) - t0;
    const bool parts = nparts > 1;
    float *dst_d2 = parts ? a.part_d2 + size_t(part) * gridDim.y * a.Q * K : a.out_dist2;
    int64_t *dst_idx = parts ? a.part_idx + size_t(part) * gridDim.y * a.Q * K : a.out_idx;

    if (blockIdx.x * BQ_CWARPS * G >= Qb) {
        if (part != 0) return;
        // every query of this block is past the cloud's valid length
        const int r0 = blockIdx.x * BQ_CWARPS * G;
        const int r1 = min(a.Q, r0 + BQ_CWARPS * G);
        const size_t e0 = (size_t(b) * a.Q + r0) * K;
        const size_t e1 = (size_t(b) * a.Q + r1) * K;
        for (size_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
            a.out_idx[e] = -1;
            a.out_dist2[e] = 0.0f;
        }
        return;
    }

    if (threadIdx.x == 0) {
        stream_init(ring, BQ_CWARPS);
        *s_err = 0;
        *s_stop = 0;
        *s_ndone = 0;
    }
    const FilterFrame fr = filter_frame(cref, min(ST_T, Nb));
    __syncthreads();

    if (warp == BQ_CWARPS) {  // producer warp: tiles strictly in input order
        const bool withhold = (a.stall & PC_STALL_TILE_STREAM) && blockIdx.x == 0 &&
                              blockIdx.y == 0 && blockIdx.z == 0;
        stream_produce<BQ_SB, false>(ring, cref, Nb, ntiles, [t0](int it) { return t0 + it; },
                                     fr, s_stop, s_err, a.timeout_ns, withhold);
        return;
    }

    const int q_warp0 = (blockIdx.x * BQ_CWARPS + warp) * G;
    const int nq = max(0, min(G, Qb - q_warp0));
    BqSlot *slots = slots_all + warp * G;
    const float *cq = a.query + size_t(b) * size_t(a.Q) * 3;
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
        const float thr = filter_threshold(a.R2, filter_query(xp, yp, zp, ax, ay, az));
        slots[g].axy = make_float4(ax, ax, ay, ay);
        slots[g].azt = make_float4(az, az, thr, __int_as_float(g));
        slots[g].raw = make_float4(x, y, z, __int_as_float(0));
    }
    __syncwarp();

    // Queries still short of K hits occupy slots [0, active); a query that
    // fills up is swapped behind them, so the hot loop checks nothing per
    // query.
    volatile int *vstop = s_stop;
    int active = nq;
    if (active == 0 && lane == 0 && atomicAdd(s_ndone, 1) + 1 == BQ_CWARPS)
        *vstop = 1;
    bool failed = false;
    for (int it = 0; it < ntiles; ++it) {
        if (__any_sync(FULL, *vstop != 0)) break;
        const int st = it % ST_STAGES;
        const WaitResult w = warp_wait(&ring.ready[st], unsigned((it / ST_STAGES) & 1),
                                       s_stop, a.timeout_ns);
        if (w != WAIT_OK) {
            failed = w == WAIT_TIMEOUT;
            break;
        }
        const int j0 = (t0 + it) * ST_T;
        const int cnt = min(ST_T, Nb - j0);
        const float4 *ck = ring.cooked_tile(st);
        const float4 *raw = ring.raw_copy(st);
        if (active > 0) {
            // the prepared points of this lane: pairs l + 32 p (points past
            // cnt are (0, 0, 0, +inf): they pass only an infinite threshold
            // and are masked exactly)
            float2 rx[BQ_R / 2], ry[BQ_R / 2], rz[BQ_R / 2], rw[BQ_R / 2];
#pragma unroll
            for (int p = 0; p < BQ_R / 2; ++p) {
                const float4 A = ck[cooked_slot<BQ_SB>(lane + 32 * p, 0)];
                const float4 Z = ck[cooked_slot<BQ_SB>(lane + 32 * p, 1)];
                rx[p] = make_float2(A.x, A.y);
                ry[p] = make_float2(A.z, A.w);
                rz[p] = make_float2(Z.x, Z.y);
                rw[p] = make_float2(Z.z, Z.w);
            }

            bool any_full = false;
            auto record = [&](BqSlot *sp, float4 axy, float4 azt) {
                const float4 q = sp->raw;
                const size_t row = size_t(b) * a.Q + q_warp0 + __float_as_int(azt.w);
                const int h = bq_record(raw, rx, ry, rz, rw, axy, azt, q,
                                        __float_as_int(q.w), j0, cnt, a.R2, K, row,
                                        dst_d2, dst_idx);
                if (lane == 0) sp->raw.w = __int_as_float(h);
                any_full |= h >= K;
            };
            // two queries per step: independent filter chains for the scheduler
            int g = 0;
            for (; g + 1 < active; g += 2) {
                BqSlot *s0 = slots + g;
                const float4 axy0 = s0[0].axy, azt0 = s0[0].azt;
                const float4 axy1 = s0[1].axy, azt1 = s0[1].azt;
                const bool t0 = filter_any8(rx, ry, rz, rw, axy0, azt0);
                const bool t1 = filter_any8(rx, ry, rz, rw, axy1, azt1);
                const bool v0 = __any_sync(FULL, t0), v1 = __any_sync(FULL, t1);
                if (v0) record(s0, axy0, azt0);
                if (v1) record(s0 + 1, axy1, azt1);
            }
            if (g < active) {
                BqSlot *s0 = slots + g;
                const float4 axy = s0->axy, azt = s0->azt;
                if (__any_sync(FULL, filter_any8(rx, ry, rz, rw, axy, azt)))
                    record(s0, axy, azt);
            }
            if (any_full) {  // rare: move full queries behind the active ones
                __syncwarp();
                if (lane == 0) {
                    int g = 0;
                    while (g < active) {
                        if (__float_as_int(slots[g].raw.w) >= K) {
                            const BqSlot t = slots[g];
                            slots[g] = slots[active - 1];
                            slots[active - 1] = t;
                            --active;
                        } else {
                            ++g;
                        }
                    }
                }
                active = __shfl_sync(FULL, active, 0);
                __syncwarp();
                if (active == 0 && lane == 0 &&
                    atomicAdd(s_ndone, 1) + 1 == BQ_CWARPS)
                    *vstop = 1;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[st]);  // stage no longer read
    }

    if (failed) {
        if (lane == 0) {
            *s_err = 1;
            *vstop = 1;
        }
        raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
    }
    // pad the unused slots with (-1, 0); after a failure every slot; rows
    // past the valid length in full.  Parts record their hit counts instead
    // (-1 after a failure); the merge pads.
    __syncwarp();
    if (parts) {
        for (int g = lane; g < nq; g += 32) {
            const BqSlot q = slots[g];
            const size_t row = size_t(b) * a.Q + q_warp0 + __float_as_int(q.azt.w);
            a.part_cnt[size_t(part) * gridDim.y * a.Q + row] =
                failed ? -1 : __float_as_int(q.raw.w);
        }
        if (part != 0) return;
    }
    const int nrows = max(0, min(G, a.Q - q_warp0));
    for (int g = nq; g < nrows; ++g) {
        const size_t row = size_t(b) * a.Q + q_warp0 + g;
        for (int e = lane; e < K; e += 32) {
            a.out_idx[row * K + e] = -1;
            a.out_dist2[row * K + e] = 0.0f;
        }
    }
    if (parts) return;
    for (int g = 0; g < nq; ++g) {
        const BqSlot q = slots[g];
        const size_t row = size_t(b) * a.Q + q_warp0 + __float_as_int(q.azt.w);
        const int hits = failed ? 0 : __float_as_int(q.raw.w);
        for (int e = hits + lane; e < K; e += 32) {
            a.out_idx[row * K + e] = -1;
            a.out_dist2[row * K + e] = 0.0f;
        }
    }
}

// The first K hits of a valid query row over the parts, in part order (a
// part covers the references after the previous part's): one warp per row.
// Slot e takes entry e - (hits of the parts before) of the part it falls
// in; past the total, (-1, 0).  A row with a stopped part is -1 throughout.
constexpr int BQ_MERGE_WARPS = 8;
__global__ void __launch_bounds__(32 * BQ_MERGE_WARPS) bq_merge_parts_kernel(const BqArgs a,
                                                                            int nparts) {
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * BQ_MERGE_WARPS + (threadIdx.x >> 5);
    const int b = blockIdx.y;
    const int B = gridDim.y;
    if (r >= valid_len(a.q_len, b, a.Q)) return;  // padded by the query kernel
    const int K = a.K;
    const size_t row = size_t(b) * a.Q + r;
    const int c = lane < nparts ? a.part_cnt[size_t(lane) * B * a.Q + row] : 0;
    const bool failed = __any_sync(FULL, c < 0);
    // inclusive prefix of the parts' hit counts over lanes 0 .. nparts - 1
    int incl = c < 0 ? 0 : c;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        const int y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
    }
    int upto[8];  // hits of parts 0 .. p, every lane
#pragma unroll
    for (int p = 0; p < 8; ++p) upto[p] = __shfl_sync(FULL, incl, p);
    const int total = upto[7];
    for (int e = lane; e < K; e += 32) {
        int64_t idx = -1;
        float d2 = 0.0f;
        if (!failed && e < total) {
            int p = 0, before = 0;
            for (; p < nparts; ++p) {
                if (e < upto[p]) break;
                before = upto[p];
            }
            const size_t src = (size_t(p) * B * a.Q + row) * K + (e - before);
            idx = a.part_idx[src];
            d2 = a.part_d2[src];
        }
        a.out_idx[row * K + e] = idx;
        a.out_dist2[row * K + e] = d2;
    }
}

}  // namespace

cudaError_t launch_ball_query(const DeviceInfo &dev, const float *query,
                              int64_t B, int64_t Q, const float *ref,
                              int64_t N, const int64_t *q_len,
                              const int64_t *r_len, float r32, int64_t K,
                              float *out_dist2, int64_t *out_idx,
                              cudaStream_t stream) {
    BqArgs a{};
    a.query = query;
    a.ref = ref;
    a.q_len = q_len;
    a.r_len = r_len;
    a.Q = static_cast<int>(Q);
    a.N = static_cast<int>(N);
    a.R2 = r32 * r32;  // fl32(fl32(r) * fl32(r)): a single float multiply
    a.K = static_cast<int>(K);
    a.out_dist2 = out_dist2;
    a.out_idx = out_idx;
    a.status = dev.status_word;
    a.timeout_ns = wait_timeout_ns();
    a.stall = debug_stall();

    // one wave of two blocks per SM, less the SMs other work holds
    const int slots = std::max(1, dev.sm_count - sm_reserve()) * 2;
    auto queries_per_warp = [&](int64_t parts) {
        const int64_t bpc_target =
            std::max<int64_t>(1, slots / std::max<int64_t>(B * parts, 1));
        return (Q + BQ_CWARPS * bpc_target - 1) / (BQ_CWARPS * bpc_target);
    };
    // Few queries against many references: a warp would hold too few queries
    // to spread each tile's cost over, so the references are split into
    // parts (blocks of the same queries, other tiles) and the parts' hits
    // merged in order (GB300, 16,384 queries vs 1M points, r = 0.01, K = 64:
    // 7 queries per warp in one part).
    const int64_t ntiles = (N + ST_T - 1) / ST_T;
    int64_t P = 1;
    const int64_t g1 = queries_per_warp(1);
    if (g1 < BQ_MIN_QUERIES_PER_WARP && ntiles >= 64)
        P = std::max<int64_t>(1, std::min<int64_t>(
                                     {BQ_MAX_PARTS,
                                      (BQ_MIN_QUERIES_PER_WARP + g1 - 1) / g1, ntiles / 16}));
    const size_t part_rows = size_t(P) * size_t(B) * size_t(Q);
    if (P > 1 && part_rows * size_t(K) * 12 > (size_t(1) << 30)) P = 1;  // scratch cap
    int64_t G = queries_per_warp(P);
    const size_t budget =
        std::min<size_t>(dev.smem_per_block_optin, dev.smem_per_sm / 2 - 2048);
    const int64_t gmax = std::max<int64_t>(
        1, int64_t((budget - bq_fixed_smem()) / (BQ_CWARPS * sizeof(BqSlot))));
    G = std::max<int64_t>(1, std::min(G, gmax));
    a.q_per_warp = static_cast<int>(G);
    const int64_t bpc = (Q + BQ_CWARPS * G - 1) / (BQ_CWARPS * G);
    const size_t smem = bq_fixed_smem() + size_t(BQ_CWARPS) * G * sizeof(BqSlot);
    cudaError_t e = cudaFuncSetAttribute(
        bq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(bpc), static_cast<unsigned>(B), static_cast<unsigned>(P));
    if (P == 1) {
        bq_kernel<<<grid, BQ_THREADS, smem, stream>>>(a);
        return cudaGetLastError();
    }
    // the parts' hits and counts in stream-ordered scratch
    const size_t rows = size_t(P) * size_t(B) * size_t(Q);
    const size_t off_d2 = (rows * size_t(K) * sizeof(int64_t) + 255) & ~size_t(255);
    const size_t off_cnt = (off_d2 + rows * size_t(K) * sizeof(float) + 255) & ~size_t(255);
    const size_t total = off_cnt + rows * sizeof(int);
    char *base = nullptr;
    e = scratch_alloc(dev, reinterpret_cast<void **>(&base), total, stream);
    if (e != cudaSuccess) return e;
    a.part_idx = reinterpret_cast<int64_t *>(base);
    a.part_d2 = reinterpret_cast<float *>(base + off_d2);
    a.part_cnt = reinterpret_cast<int *>(base + off_cnt);
    bq_kernel<<<grid, BQ_THREADS, smem, stream>>>(a);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
        const dim3 gm(static_cast<unsigned>((Q + BQ_MERGE_WARPS - 1) / BQ_MERGE_WARPS),
                      static_cast<unsigned>(B));
        bq_merge_parts_kernel<<<gm, 32 * BQ_MERGE_WARPS, 0, stream>>>(a, int(P));
        e = cudaGetLastError();
    }
    const cudaError_t f = scratch_free(base, stream);
    return e != cudaSuccess ? e : f;
}

}  // namespace pcn
