// pc_device.cuh -- device primitives shared by the FPS, kNN and Ball Query
// kernels: the non-contracted squared distance, warp reductions, and inline
// PTX for mbarriers, TMA bulk copies, clusters and bounded waits (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pcn {

// ---------------------------------------------------------------------------
// Squared distance s = ((dx*dx + dy*dy) + dz*dz), each operation rounded to
// nearest even on its own (no FMA), as the mps-pointops project page's
// "How the kernels work" section states for FPS and kNN and as the
// "Numerical contracts" page's s32 requires for all three operators.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sqdist(float ax, float ay, float az,
                                        float bx, float by, float bz) {
    float dx = __fsub_rn(ax, bx);
    float dy = __fsub_rn(ay, by);
    float dz = __fsub_rn(az, bz);
    return __fadd_rn(__fadd_rn(__fmul_rn(dx, dx), __fmul_rn(dy, dy)),
                     __fmul_rn(dz, dz));
}

// The smallest of three floats in one instruction (three-operand min.f32,
// sm_100 and later).  A NaN operand is ignored unless all three are NaN, as
// with fminf; the filters use it only on values that are never NaN.
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed f32x2 arithmetic in PTX.  add2_rn is one round-to-nearest-even
// addition per half.  Squares are NOT written as mul.rn.f32x2: ptxas fuses a
// single-use packed multiply into the packed add that consumes it (an FMA,
// one rounding instead of two) even with an explicit .rn modifier and
// --fmad=false.  A square is therefore computed as fma.rn.f32x2(d, d, z) with
// z = (-0, -0) supplied at run time: d*d + (-0) is exactly d*d (also for a
// zero product, +0 + -0 = +0), so the FMA returns RN(d*d), the same float as
// a separately rounded multiply; and since the addend is not a compile-time
// constant the compiler cannot rewrite the FMA into a fusable multiply.
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// RN(a * a) per half; `negzero` must hold (-0.0f, -0.0f) at run time.
__device__ __forceinline__ float2 sq2_rn(float2 a, float2 negzero) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rz, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rz, {%4, %5};\n\t"
        "fma.rn.f32x2 rd, ra, ra, rz;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(negzero.x), "f"(negzero.y));
    return d;
}

// Two references (packed in the .x/.y halves) against one point whose
// coordinates are given NEGATED: d = x + (-q) is the same float as -(q - x)
// under round-to-nearest-even, and the square removes the sign, so each half
// equals sqdist() bit for bit: ((dx*dx + dy*dy) + dz*dz), five roundings.
__device__ __forceinline__ float2 sqdist2(float2 x, float2 y, float2 z,
                                          float2 nqx, float2 nqy, float2 nqz,
                                          float2 negzero) {
    const float2 dx = add2_rn(x, nqx);
    const float2 dy = add2_rn(y, nqy);
    const float2 dz = add2_rn(z, nqz);
    return add2_rn(add2_rn(sq2_rn(dx, negzero), sq2_rn(dy, negzero)),
                   sq2_rn(dz, negzero));
}

__device__ __forceinline__ unsigned lane_id() {
    unsigned r;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned r;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
    return r;
}

// Barrier `id` (1..15) over the first `nthreads` threads that reach it (a
// multiple of 32: whole warps).
__device__ __forceinline__ void named_barrier_sync(unsigned id, unsigned nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier (shared::cta) and TMA bulk copies global -> shared.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      unsigned bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Wait for phase `parity` of `bar` to complete, at most `timeout_ns`.
// Returns false if the bound ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar,
                                                  unsigned parity,
                                                  uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (;;) {
        #pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// 1-D bulk copy (TMA) of `bytes` bytes global -> shared, completing on `bar`
// as transaction bytes.  dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src,
                                         unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes "
        "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 4-byte asynchronous copy global -> shared (for unaligned tile edges).
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)),
                 "l"(src)
                 : "memory");
}

// Make `bar` track completion of this thread's prior cp.async operations
// (the pending count is raised now and lowered when they land).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.shared.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread block clusters.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_ctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ unsigned cluster_nctarank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Address of the same shared variable in cluster block `rank`.
__device__ __forceinline__ uint32_t map_shared_rank(const void *p,
                                                    unsigned rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(r)
                 : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a,
                                              uint32_t b, uint32_t c,
                                              uint32_t d) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                 "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Asynchronous stores into another block's shared memory (distributed shared
// memory) that signal completion as transaction bytes on an mbarrier in that
// block.  Both addresses are shared::cluster addresses (map_shared_rank).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a,
                                            uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 "
        "[%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
        "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t v,
                                             uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 "
        "[%0], %1, [%2];" ::"r"(addr),
        "r"(v), "r"(bar)
        : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from this block's shared memory to the shared memory of a block of the
// cluster, completing as transaction bytes on an mbarrier in that block.
// dst and bar are shared::cluster addresses (map_shared_rank).  The source
// must have been made visible to the async proxy (fence_proxy_async_smem
// after the writes) and must not be written again before
// bulk_wait_read_all() in the issuing thread.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst, const void *src,
                                                     unsigned bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes "
        "[%0], [%1], %2, [%3];" ::"r"(dst),
        "r"(smem_u32(src)), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the issuing thread's committed bulk copies have read their sources
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// the issuing thread's committed bulk copies are complete
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// try_wait with cluster-scope acquire: data that other blocks of the cluster
// delivered with st.async is visible once the phase completes.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar,
                                                      unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar,
                                                          unsigned parity,
                                                          uint64_t timeout_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// Full cluster barrier: every thread of every block of the cluster arrives
// (release) and waits (acquire).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// ---------------------------------------------------------------------------
// Global memory accesses with explicit memory-model semantics.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t *p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t *p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v)
                 : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Record the first device-side error in the library's status word.
__device__ __forceinline__ void raise_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Warp reductions of (hi, lo) pairs in lexicographic order.
// ---------------------------------------------------------------------------
// Returns the largest hi over the warp and, among lanes holding it, the
// smallest lo.
__device__ __forceinline__ void warp_argmax_hi_min_lo(unsigned hi, unsigned lo,
                                                      unsigned &best_hi,
                                                      unsigned &best_lo) {
    best_hi = __reduce_max_sync(0xffffffffu, hi);
    best_lo = __reduce_min_sync(0xffffffffu, hi == best_hi ? lo : 0xffffffffu);
}

}  // namespace pcn
