// pc_tiles.cuh -- double-buffered staging of reference tiles into shared
// memory for the kNN and Ball Query kernels.
//
// A tile is `cnt` consecutive reference points (x, y, z float32, 12 bytes
// each) of one cloud.  Clouds start at any 4-byte boundary (B clouds of N
// points are packed back to back), so a tile's bytes [g0, g1) are split into
//   - the 16-byte-aligned interior, copied by one TMA bulk copy
//     (cp.async.bulk, completes as transaction bytes on the stage mbarrier),
//   - at most three 4-byte words before it and three after it, copied by
//     4-byte cp.async whose completion the same mbarrier tracks.
// In shared memory the tile keeps its global alignment modulo 16: byte 0 of
// the buffer corresponds to global address (g0 & ~15), so point i of the
// tile starts at float index tile_float_offset(g0) + 3*i.
#pragma once

#include "pc_device.cuh"

namespace pcn {

// Bytes reserved per tile buffer for `T` points (16-byte multiple).
__host__ __device__ constexpr unsigned tile_buffer_bytes(unsigned T) {
    return ((12u * T + 16u) + 15u) & ~15u;
}

__device__ __forceinline__ unsigned tile_float_offset(const float *g0) {
    return static_cast<unsigned>(reinterpret_cast<uintptr_t>(g0) & 15u) >> 2;
}

// Called by ONE thread.  Copies points [0, cnt) starting at `gsrc` into the
// 16-byte-aligned buffer `buf`; completion is signalled on `bar`, which must
// have been initialised with an arrival count of 1.
__device__ __forceinline__ void issue_tile(float *buf, const float *gsrc,
                                           int cnt, uint64_t *bar) {
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(gsrc);
    const uintptr_t g1 = g0 + 12ull * static_cast<unsigned>(cnt);
    const uintptr_t base = g0 & ~uintptr_t(15);
    const uintptr_t a0 = (g0 + 15) & ~uintptr_t(15);
    const uintptr_t a1 = g1 & ~uintptr_t(15);
    char *b = reinterpret_cast<char *>(buf);
    const uintptr_t head_end = a0 < g1 ? a0 : g1;
    for (uintptr_t a = g0; a < head_end; a += 4)
        cp_async_4(b + (a - base), reinterpret_cast<const void *>(a));
    const uintptr_t tail_beg = a1 > head_end ? a1 : head_end;
    for (uintptr_t a = tail_beg; a < g1; a += 4)
        cp_async_4(b + (a - base), reinterpret_cast<const void *>(a));
    cp_async_mbar_arrive(bar);
    const unsigned bulk = a1 > a0 ? static_cast<unsigned>(a1 - a0) : 0u;
    // the buffer was last read through the generic proxy; order those reads
    // before the async-proxy writes below
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, bulk);
    if (bulk)
        bulk_g2s(b + (a0 - base), reinterpret_cast<const void *>(a0), bulk, bar);
}

// Called by ONE thread.  Copies cnt >= 1 points of 16 bytes from the
// 16-byte-aligned `gsrc` into `buf` with one bulk copy; completion is
// signalled on `bar` (arrival count 1).
__device__ __forceinline__ void issue_tile16(float *buf, const float *gsrc, int cnt,
                                             uint64_t *bar) {
    const unsigned bytes = 16u * static_cast<unsigned>(cnt);
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(buf, gsrc, bytes, bar);
}

// ---------------------------------------------------------------------------
// Ring of STAGES tile buffers shared by the consumer warps of a block and
// filled by one producer thread.  full[s] (count 1 + transaction bytes)
// completes when tile data has landed; empty[s] (count = consumer warps)
// completes when every consumer warp has copied the tile into registers.
// Consumers therefore drift freely by up to STAGES - 1 tiles instead of
// meeting at a block barrier every tile.
// ---------------------------------------------------------------------------
struct TileRing {
    unsigned char *base;  // STAGES buffers of `bytes` bytes, 16-byte aligned
    unsigned bytes;
    uint64_t *full;
    uint64_t *empty;
    __device__ __forceinline__ float *buf(int s) const {
        return reinterpret_cast<float *>(base + size_t(s) * bytes);
    }
};

// Status of a bounded wait that may also be told to stop.
enum WaitResult { WAIT_OK = 0, WAIT_TIMEOUT = 1, WAIT_STOPPED = 2 };

// Wait for phase `parity` of `bar`; give up when `*stop` becomes non-zero
// (checked every 64 polls) or after timeout_ns.
__device__ __forceinline__ WaitResult mbar_wait_or_stop(uint64_t *bar,
                                                        unsigned parity,
                                                        const volatile int *stop,
                                                        uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return WAIT_OK;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return WAIT_OK;
        if (stop && *stop) return WAIT_STOPPED;
        if (global_timer_ns() - t0 > timeout_ns) return WAIT_TIMEOUT;
    }
}

// Producer loop, run by ONE thread.  Tile `it` (it = 0..ntiles-1) covers
// points [tile_at(it) * T, ...) of the cloud starting at `cref`.  Stops early
// when `*stop` becomes non-zero; on a timeout it raises *err.  Before
// returning it waits (bounded) until every copy it issued has landed, so no
// copy is in flight when the block exits.  withhold_first (a testing hook)
// skips the first tile's copy altogether: the waits for it run out.
template <int STAGES, class TileAt>
__device__ __forceinline__ void ring_produce(const TileRing &ring,
                                             const float *cref, int N, int T,
                                             int ntiles, TileAt tile_at,
                                             volatile int *stop,
                                             volatile int *err,
                                             uint64_t timeout_ns,
                                             bool withhold_first = false) {
    int issued = 0;
    for (int it = 0; it < ntiles; ++it) {
        const int st = it % STAGES;
        if (it >= STAGES) {
            const WaitResult w = mbar_wait_or_stop(
                &ring.empty[st], unsigned((it / STAGES - 1) & 1), stop,
                timeout_ns);
            if (w == WAIT_TIMEOUT) *err = 1;
            if (w != WAIT_OK) break;
        }
        if (*stop || *err) break;
        const int j0 = tile_at(it) * T;
        if (!(withhold_first && it == 0))
            issue_tile(ring.buf(st), cref + size_t(j0) * 3, min(T, N - j0),
                       &ring.full[st]);
        issued = it + 1;
    }
    for (int st = 0; st < STAGES; ++st) {
        // last tile issued into stage st
        const int last = issued - 1 - ((issued - 1 - st) % STAGES + STAGES) % STAGES;
        if (issued > 0 && last >= 0 && last % STAGES == st)
            mbar_wait_bounded(&ring.full[st], unsigned((last / STAGES) & 1),
                              timeout_ns);
    }
}

}  // namespace pcn
