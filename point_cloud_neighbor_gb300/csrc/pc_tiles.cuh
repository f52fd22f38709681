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

}  // namespace pcn
