// pc_stream.cuh -- reference-tile streaming with producer-side preparation,
// for the lane-per-query kNN and Ball Query kernels.
//
// A block has CW consumer warps and one producer warp.  The producer warp
// streams reference tiles of ST_T points:
//   1. its lane 0 copies raw tiles (x, y, z float32) with TMA (issue_tile of
//      pc_tiles.cuh) into a private ring of ST_RAW_STAGES buffers, up to
//      ST_RAW_STAGES tiles ahead of its own preparation;
//   2. once a raw tile has landed and the stage it goes to has been released
//      by every consumer warp, the whole warp "cooks" it into the stage: the
//      centred coordinates and w' of the filter of pc_filter.cuh, packed for
//      the paired instructions, two points (a "pair" p) per 32 bytes,
//          A(p) = (x'_2p, x'_2p+1, y'_2p, y'_2p+1)
//          Z(p) = (z'_2p, z'_2p+1, w'_2p, w'_2p+1),
//      and a copy of the raw coordinates (x, y, z, 0) per point for the
//      exact path; points past the tile's end get (0, 0, 0, +inf): they pass
//      the filter only against an infinite threshold and are masked exactly
//      (t' = +inf there; every other t' is finite or -inf, see pc_filter.cuh);
//   3. all 32 producer lanes arrive on the stage's `ready` barrier, and the
//      raw buffer is refilled with the tile ST_RAW_STAGES further on.
// The raw ring never waits on the consumers, so the producer can run up to
// ST_STAGES cooked tiles ahead of the slowest consumer warp.
//
// Layout of a stage: 16-byte slots in rows of 8 (128 bytes, one pass over
// the 32 banks).  Step s = the 8 points 8s .. 8s + 7 = pairs 4s .. 4s + 3;
// its cooked row holds A and Z of pair 4s + u at slots 2u and 2u + 1, XORed
// with the low SB bits of s (shifted to the top of the 3-bit slot index), and
// its raw row point 8s + r at slot r XOR (s & 7).  A warp whose lanes all
// read step s gets broadcasts either way; lanes reading the same slot of
// different steps (the per-lane slow paths) land on 2^SB different bank
// groups instead of one.  The consumers' hot loop walks 2^SB steps per
// iteration so that its slot offsets are compile-time constants.  Consumers wait
// on `ready`, read the cooked tile (every lane reads the same 16 bytes:
// shared-memory broadcasts) and, on their rare slow paths, the raw copy;
// then each consumer warp arrives on `empty`, which the producer waits on
// before it reuses the stage.  Every wait is bounded.
#pragma once

#include "pc_device.cuh"
#include "pc_filter.cuh"
#include "pc_tiles.cuh"

namespace pcn {

constexpr int ST_T = 256;  // points per tile
constexpr int ST_STAGES = 8;      // cooked stages (shared with the consumers)
constexpr int ST_RAW_STAGES = 3;  // TMA landing buffers (producer only)
// a raw tile: ST_T points of 12 bytes (plus alignment), or of 16 bytes
// (x, y, z, original index) for clouds in a spatial order
constexpr unsigned ST_RAW = tile_buffer_bytes(ST_T) > ST_T * 16u ? tile_buffer_bytes(ST_T)
                                                                  : ST_T * 16u;
constexpr unsigned ST_COOKED = (ST_T / 2) * 32;
constexpr unsigned ST_COPY = ST_T * 16;  // raw coordinates, 16 bytes a point
constexpr unsigned ST_STAGE = ST_COOKED + ST_COPY;

static_assert(ST_RAW % 16 == 0 && ST_STAGE % 16 == 0, "buffers stay 16-byte aligned");

struct StreamRing {
    unsigned char *stage;  // ST_STAGES x (cooked, raw copy)
    unsigned char *raw;    // ST_RAW_STAGES x ST_RAW bytes
    uint64_t *raw_full;    // [ST_RAW_STAGES] count 1 + transaction bytes
    uint64_t *ready;       // [ST_STAGES] count 32 (the producer warp)
    uint64_t *empty;       // [ST_STAGES] count = consumer warps
    __device__ __forceinline__ const float4 *cooked_tile(int s) const {
        return reinterpret_cast<const float4 *>(stage + size_t(s) * ST_STAGE);
    }
    // (x, y, z, 0) of point i of the tile at [raw_slot(i)]
    __device__ __forceinline__ const float4 *raw_copy(int s) const {
        return reinterpret_cast<const float4 *>(stage + size_t(s) * ST_STAGE + ST_COOKED);
    }
    __device__ __forceinline__ float *raw_tile(int r) const {
        return reinterpret_cast<float *>(raw + size_t(r) * ST_RAW);
    }
};

// Shared memory of the rings plus 16 bytes of flags (error, stop, warps
// done), rounded up to 16 bytes so that whatever follows may hold 16-byte
// vectors.
__host__ __device__ constexpr size_t stream_smem_bytes() {
    return (size_t(ST_STAGES) * ST_STAGE + size_t(ST_RAW_STAGES) * ST_RAW +
            (ST_RAW_STAGES + 2 * ST_STAGES) * 8 + 16 + 15) & ~size_t(15);
}
static_assert(stream_smem_bytes() % 16 == 0, "16-byte aligned end");

// Carve the rings out of `smem` (16-byte aligned); returns the flag words.
__device__ __forceinline__ int *stream_carve(unsigned char *smem, StreamRing &r) {
    r.stage = smem;
    r.raw = smem + size_t(ST_STAGES) * ST_STAGE;
    r.raw_full = reinterpret_cast<uint64_t *>(r.raw + size_t(ST_RAW_STAGES) * ST_RAW);
    r.ready = r.raw_full + ST_RAW_STAGES;
    r.empty = r.ready + ST_STAGES;
    return reinterpret_cast<int *>(r.empty + ST_STAGES);
}

// Slot of A (h = 0) or Z (h = 1) of pair p in a cooked tile (SB = 2 or 3
// swizzle bits), and of point i in a raw copy.
template <int SB>
__host__ __device__ __forceinline__ int cooked_slot(int p, int h) {
    static_assert(SB >= 1 && SB <= 3, "1 to 3 swizzle bits");
    return ((p >> 2) << 3) |
           ((((p & 3) << 1) | h) ^ (((p >> 2) & ((1 << SB) - 1)) << (3 - SB)));
}
__host__ __device__ __forceinline__ int raw_slot(int i) {
    return (i & ~7) | ((i & 7) ^ ((i >> 3) & 7));
}

// Called by thread 0 before the block's first __syncthreads.
__device__ __forceinline__ void stream_init(const StreamRing &r, int consumer_warps) {
    for (int s = 0; s < ST_RAW_STAGES; ++s) mbar_init(&r.raw_full[s], 1);
    for (int s = 0; s < ST_STAGES; ++s) {
        mbar_init(&r.ready[s], 32);
        mbar_init(&r.empty[s], consumer_warps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Warp-uniform bounded wait (every lane polls; the result is agreed on).
__device__ __forceinline__ WaitResult warp_wait(uint64_t *bar, unsigned parity,
                                                const volatile int *stop,
                                                uint64_t timeout_ns) {
    const WaitResult w = mbar_wait_or_stop(bar, parity, stop, timeout_ns);
    if (__all_sync(0xffffffffu, w == WAIT_OK)) return WAIT_OK;
    return __any_sync(0xffffffffu, w == WAIT_TIMEOUT) ? WAIT_TIMEOUT : WAIT_STOPPED;
}

// The producer warp.  Tile `it` covers points [tile_at(it) * ST_T, ...) of
// the cloud at `cref` (N valid points): (x, y, z) float triples, or with F4
// 16-byte points (x, y, z, original index bits) starting 16-byte aligned,
// whose index goes to the fourth component of the raw copy (0 otherwise).
// Stops when *stop becomes non-zero; a timeout raises *err.  Before
// returning it waits (bounded) for every raw copy it issued, so none is in
// flight when the block exits.  withhold_first (a testing hook) skips the
// first tile's copy altogether: its wait, and the consumers', run out.
template <int SB, bool F4, class TileAt>
__device__ __forceinline__ void stream_produce(const StreamRing &ring,
                                               const float *cref, int N,
                                               int ntiles, TileAt tile_at,
                                               FilterFrame fr,
                                               volatile int *stop,
                                               volatile int *err,
                                               uint64_t timeout_ns,
                                               bool withhold_first = false) {
    const int lane = static_cast<int>(lane_id());
    const float inf = __int_as_float(0x7f800000);
    int issued = 0, landed = 0;
    constexpr int PS = F4 ? 4 : 3;  // floats per point
    auto issue = [&](int t, int slot) {
        const int j0 = tile_at(t) * ST_T;
        if (F4)
            issue_tile16(ring.raw_tile(slot), cref + size_t(j0) * 4, min(ST_T, N - j0),
                         &ring.raw_full[slot]);
        else
            issue_tile(ring.raw_tile(slot), cref + size_t(j0) * 3, min(ST_T, N - j0),
                       &ring.raw_full[slot]);
    };
    if (lane == 0)
        for (; issued < ntiles && issued < ST_RAW_STAGES; ++issued)
            if (!(withhold_first && issued == 0)) issue(issued, issued);
    issued = __shfl_sync(0xffffffffu, issued, 0);
    for (int it = 0; it < ntiles; ++it) {
        const int st = it % ST_STAGES, rs = it % ST_RAW_STAGES;
        const WaitResult wr = warp_wait(&ring.raw_full[rs],
                                        unsigned((it / ST_RAW_STAGES) & 1), nullptr,
                                        timeout_ns);
        if (wr != WAIT_OK) {
            if (lane == 0) *err = 1;
            break;
        }
        landed = it + 1;
        if (it >= ST_STAGES) {
            const WaitResult w = warp_wait(&ring.empty[st],
                                           unsigned((it / ST_STAGES - 1) & 1), stop,
                                           timeout_ns);
            if (w == WAIT_TIMEOUT && lane == 0) *err = 1;
            if (w != WAIT_OK) break;
        }
        if (__any_sync(0xffffffffu, *stop != 0 || *err != 0)) break;
        const int j0 = tile_at(it) * ST_T;
        const int cnt = min(ST_T, N - j0);
        const float *src =
            ring.raw_tile(rs) + (F4 ? 0u : tile_float_offset(cref + size_t(j0) * 3));
        float4 *dst = reinterpret_cast<float4 *>(ring.stage + size_t(st) * ST_STAGE);
        float4 *copy = reinterpret_cast<float4 *>(ring.stage + size_t(st) * ST_STAGE +
                                                  ST_COOKED);
#pragma unroll
        for (int u = 0; u < ST_T / 64; ++u) {
            const int p = lane + 32 * u;
            float c[2][4], r[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int i = 2 * p + h;
                r[h][3] = 0.f;
                if (i < cnt) {
                    r[h][0] = src[PS * i];
                    r[h][1] = src[PS * i + 1];
                    r[h][2] = src[PS * i + 2];
                    if (F4) r[h][3] = src[PS * i + 3];
                    float xp = __fsub_rn(r[h][0], fr.cx);
                    float yp = __fsub_rn(r[h][1], fr.cy);
                    float zp = __fsub_rn(r[h][2], fr.cz);
                    c[h][3] = filter_ref(xp, yp, zp);
                    c[h][0] = xp;
                    c[h][1] = yp;
                    c[h][2] = zp;
                } else {
                    r[h][0] = r[h][1] = r[h][2] = 0.f;
                    c[h][0] = c[h][1] = c[h][2] = 0.f;
                    c[h][3] = inf;
                }
            }
            dst[cooked_slot<SB>(p, 0)] = make_float4(c[0][0], c[1][0], c[0][1], c[1][1]);
            dst[cooked_slot<SB>(p, 1)] = make_float4(c[0][2], c[1][2], c[0][3], c[1][3]);
            copy[raw_slot(2 * p)] = make_float4(r[0][0], r[0][1], r[0][2], r[0][3]);
            copy[raw_slot(2 * p + 1)] = make_float4(r[1][0], r[1][1], r[1][2], r[1][3]);
        }
        __syncwarp();  // every lane has read raw buffer rs
        if (lane == 0 && issued < ntiles) issue(issued, rs);
        if (issued < ntiles) ++issued;
        mbar_arrive(&ring.ready[st]);
    }
    // raw copies issued but never waited for must land before the block exits
    for (int t = landed; t < issued; ++t)
        mbar_wait_bounded(&ring.raw_full[t % ST_RAW_STAGES],
                          unsigned((t / ST_RAW_STAGES) & 1), timeout_ns);
}

// The filter of one query (broadcast operands a = (-2q', -2q') per axis)
// against points 2p .. 2p + 2v - 1 of a cooked tile: bit h of the result
// (h < 2v) is set when point 2p + h may satisfy the selection bound.
template <int SB, int V>
__device__ __forceinline__ unsigned stream_mask(const float4 *ck, int p, float2 ax,
                                                float2 ay, float2 az, float thr) {
    unsigned m = 0;
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const float4 A = ck[cooked_slot<SB>(p + u, 0)];
        const float4 Z = ck[cooked_slot<SB>(p + u, 1)];
        float2 v = __ffma2_rn(make_float2(A.x, A.y), ax, make_float2(Z.z, Z.w));
        v = __ffma2_rn(make_float2(A.z, A.w), ay, v);
        v = __ffma2_rn(make_float2(Z.x, Z.y), az, v);
        m |= (v.x <= thr ? 1u : 0u) << (2 * u);
        m |= (v.y <= thr ? 1u : 0u) << (2 * u + 1);
    }
    return m;
}

}  // namespace pcn
