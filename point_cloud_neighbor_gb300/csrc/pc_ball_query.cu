// pc_ball_query.cu -- dense first-K Ball Query on sm_103a.
//
// Operator (mps-pointops project page, "Ball Query: first K within a
// radius"; "Numerical contracts", "Selection and output"): with
// R2 = fl32(fl32(r) * fl32(r)), reference j is accepted iff s < R2; the
// first K accepted indices in input order are returned with their squared
// distances, unused slots hold (-1, 0).
//
// Design (one launch, no scratch memory):
//  * A block has BQ_CWARPS consumer warps and one producer warp; each lane of
//    a consumer warp owns one query (its filter constants -2q' in packed
//    registers, its threshold, its hit count).  The producer streams the
//    cloud's reference tiles strictly in input order and prepares them
//    (pc_stream.cuh): centred coordinates and w' packed two points per 32
//    bytes.
//  * The hot loop: per step, a lane evaluates the conservative filter of
//    pc_filter.cuh for 8 points (three packed FMAs per two points, operands
//    read as shared-memory broadcasts) against its threshold.  No vote and no
//    per-query shared state: 8 independent FMA chains per step per lane.
//  * On a pass (rare) the lane recomputes which of the 8 points passed,
//    computes their exact s32 from the raw tile and appends the hits in
//    input order straight to its output row; at K hits its threshold becomes
//    -inf.  When every query of a block is full a stop flag ends the block:
//    the producer stops issuing tiles (after letting its copies in flight
//    land) and the consumers leave the tile loop.
#include "pc_device.cuh"
#include "pc_filter.cuh"
#include "pc_internal.h"
#include "pc_stream.cuh"
#include "pc_tiles.cuh"

#include <algorithm>

namespace pcn {
namespace {

constexpr int BQ_CWARPS = 8;
constexpr int BQ_THREADS = 32 * (BQ_CWARPS + 1);
constexpr unsigned FULL = 0xffffffffu;

struct BqArgs {
    const float *query;
    const float *ref;
    const int64_t *q_len;  // valid queries per cloud (NULL: Q)
    const int64_t *r_len;  // valid references per cloud (NULL: N)
    int Q, N;
    float R2;
    int K;
    float *out_dist2;
    int64_t *out_idx;
    int *status;
    uint64_t timeout_ns;
};

// Valid length of cloud b: lens[b] clamped to [0, full], or full.
__device__ __forceinline__ int valid_len(const int64_t *lens, int b, int full) {
    if (lens == nullptr) return full;
    const int64_t v = lens[b];
    return v < 0 ? 0 : (v > full ? full : static_cast<int>(v));
}

__global__ void __launch_bounds__(BQ_THREADS, 3) bq_kernel(const BqArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int K = a.K;
    const float inf = __int_as_float(0x7f800000);

    StreamRing ring;
    int *flags = stream_carve(smem, ring);
    int *s_err = flags, *s_stop = flags + 1, *s_ndone = flags + 2;

    const float *cref = a.ref + size_t(b) * size_t(a.N) * 3;
    const int Nb = valid_len(a.r_len, b, a.N);
    const int Qb = valid_len(a.q_len, b, a.Q);
    const int ntiles = (Nb + ST_T - 1) / ST_T;
    const int q0 = blockIdx.x * BQ_CWARPS * 32;

    if (q0 >= Qb) {
        // every query of this block is past the cloud's valid length
        const int r1 = min(a.Q, q0 + BQ_CWARPS * 32);
        const size_t e0 = (size_t(b) * a.Q + q0) * K;
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

    if (warp == BQ_CWARPS) {  // producer warp
        stream_produce(ring, cref, Nb, ntiles, [](int it) { return it; }, fr,
                       s_stop, s_err, a.timeout_ns);
        return;
    }

    const int qi = q0 + warp * 32 + lane;
    const bool valid = qi < Qb;
    float qx = 0.f, qy = 0.f, qz = 0.f;
    if (valid) {
        const float *p = a.query + (size_t(b) * a.Q + qi) * 3;
        qx = p[0];
        qy = p[1];
        qz = p[2];
    }
    const float xp = __fsub_rn(qx, fr.cx), yp = __fsub_rn(qy, fr.cy),
                zp = __fsub_rn(qz, fr.cz);
    const float2 ax = make_float2(-2.0f * xp, -2.0f * xp);
    const float2 ay = make_float2(-2.0f * yp, -2.0f * yp);
    const float2 az = make_float2(-2.0f * zp, -2.0f * zp);
    float thr = valid ? filter_threshold(a.R2, filter_norm2(xp, yp, zp)) : -inf;
    const size_t row = size_t(b) * a.Q + qi;
    int hits = 0;
    bool done = !valid;
    bool reported = false;
    volatile int *vstop = s_stop;
    if (__all_sync(FULL, done)) {
        reported = true;
        if (lane == 0 && atomicAdd(s_ndone, 1) + 1 == BQ_CWARPS) *vstop = 1;
    }

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
        if (!__all_sync(FULL, done)) {
            const float4 *ck = ring.cooked_tile(st);
            const int j0 = it * ST_T;
            const int cnt = min(ST_T, Nb - j0);
            const float *raw =
                ring.raw_tile(st) + tile_float_offset(cref + size_t(j0) * 3);
            const int npairs = (cnt + 1) >> 1;
            for (int p = 0; p < npairs; p += 4) {
                if (!stream_any<4>(ck, p, ax, ay, az, thr)) continue;
                unsigned m = stream_mask<4>(ck, p, ax, ay, az, thr);
                while (m) {  // points in increasing index order
                    const int i = 2 * p + __ffs(m) - 1;
                    m &= m - 1;
                    if (i >= cnt || hits >= K) continue;
                    const float sv = sqdist(qx, qy, qz, raw[3 * i], raw[3 * i + 1],
                                            raw[3 * i + 2]);
                    if (sv < a.R2) {
                        a.out_idx[row * K + hits] = j0 + i;
                        a.out_dist2[row * K + hits] = sv;
                        if (++hits == K) {
                            done = true;
                            thr = -inf;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[st]);  // tile no longer read
        if (!reported && __all_sync(FULL, done)) {
            reported = true;
            if (lane == 0 && atomicAdd(s_ndone, 1) + 1 == BQ_CWARPS) *vstop = 1;
        }
    }

    if (failed) {
        if (lane == 0) {
            *s_err = 1;
            *vstop = 1;
        }
        raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
        hits = 0;
    }
    (void)inf;
    // pad the unused slots with (-1, 0); rows past the valid length in full
    if (qi < a.Q) {
        for (int e = valid ? hits : 0; e < K; ++e) {
            a.out_idx[row * K + e] = -1;
            a.out_dist2[row * K + e] = 0.0f;
        }
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
    (void)dev.smem_per_sm;
    const size_t smem = stream_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(
        bq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t per_block = int64_t(BQ_CWARPS) * 32;
    dim3 grid(static_cast<unsigned>((Q + per_block - 1) / per_block),
              static_cast<unsigned>(B));
    bq_kernel<<<grid, BQ_THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pcn
