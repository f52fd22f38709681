// pc_fps.cu -- farthest point sampling on sm_103a, all steps in one launch.
//
// Operator (mps-pointops project page, "Farthest point sampling" and
// "Contracts"): c_0 = start_idx; m_j(t) = min_{u<=t} s(x_j, x_{c_u});
// c_{t+1} = the smallest j attaining max_l m_l(t).
//
// Every point's coordinates and running minimum m_j stay in registers of the
// thread that owns it for the whole launch (PPT points per thread, packed in
// pairs for the f32x2 instructions), so a step reads no memory except the new
// center.  Few fat threads (about eight warps per block) keep the per-step
// reductions and barriers short.  Per step:
//   1. each thread updates its m_j with the previous center and keeps its own
//      (max m, smallest j) -- points are visited in increasing j, so a strict
//      ">" keeps the smallest index on a tie;
//   2. a warp reduces the key (bits(m) + 1, j) with two redux.sync
//      instructions (max of the first half, then min j among the lanes that
//      hold it); warp leaders publish to shared memory;
//   3. warp 0 reduces the block's candidates and looks the winner's
//      coordinates up in the block's shared-memory copy of its points;
//   4. blocks of a cloud exchange their candidates:
//      - BLOCK schedule (one block per cloud): nothing to exchange;
//      - CLUSTER schedule (one thread block cluster per cloud), by default in
//        rounds of several centers per exchange (fps_rounds_kernel: each
//        warp lists its best points and bounds the rest, and every block
//        certifies the same run of centers from the cloud's lists); one
//        center per exchange (pc_fps_set_batched(0)): warp 0 sends
//        the candidate (key, coordinates) into slot [step parity][its rank]
//        of every block of the cluster with st.async, which completes as
//        transaction bytes on that block's own mbarrier for this step
//        parity; each block waits only on its local mbarrier (one-way
//        latency, no cluster-wide barrier) and every warp reduces the
//        cluster's slots itself.  Slots and mbarriers are double buffered by
//        step parity: a block can only send step t+2 after every block sent
//        step t+1, which each does after reading step t;
//      - GRID schedule (cooperative launch, several blocks per cloud): each
//        block writes one 64-bit word [bits(m)+1 : 31 | 2^24-1-j : 24 |
//        step mod 512 : 9] into its slot of the caller's workspace; warp 0
//        of every block polls the cloud's slots until all carry this step's
//        tag, reduces them, and reads the winner's coordinates from the
//        input.  Every wait is bounded (timeout -> status word, -1 outputs).
// Points are (bits(m) + 1) so that a block without points (key 0) never
// wins; once every m is 0 the smallest index, 0, wins, which reproduces
// "remaining slots repeat index 0".
#include "pc_device.cuh"
#include "pc_internal.h"

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

namespace pcn {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int FPS_MAX_CLUSTER = 16;
constexpr int FPS_GRID_MAX_N = 1 << 24;  // index field of the exchange word
constexpr int FPS_CAND_BYTES = 20;       // key, index, x, y, z sent per block
constexpr int CG_SLOT_WORDS = 16;        // a cluster's four words, one 128-byte line

// Threads per block a kernel with PPT points per thread may use: the points'
// registers (4 per point) must fit next to the working set.
__host__ __device__ constexpr int fps_max_threads(int ppt) {
    return ppt <= 8 ? 1024 : ppt <= 16 ? 512 : ppt <= 24 ? 384 : 256;
}

struct FpsArgs {
    const float *xyz;
    int N, npoint, start;
    int64_t *out;
    int chunk;     // points per block
    int nblocks;   // blocks per cloud (cluster size or grid blocks per cloud)
    int cs;        // two-level GRID: blocks per cluster
    int ncl;       // two-level GRID: clusters per cloud
    uint64_t *slots;
    int *status;
    uint64_t timeout_ns;
    int stall;      // PC_STALL_* testing flags
    float negzero;  // -0.0f, see sq2_rn
};

struct __align__(16) ClusterSlot {
    unsigned hi, j;
    float x, y;
    float z, pad0, pad1, pad2;
};

__host__ __device__ constexpr size_t fps_coords_bytes(int chunk) {
    return (size_t(chunk) * 12 + 15) & ~size_t(15);
}

// The points of one thread: point p of the thread is j_first + p * T, packed
// in pairs (p = 2i, 2i+1) for the f32x2 instructions.
template <int PPT>
struct ThreadPoints {
    float2 x[PPT / 2], y[PPT / 2], z[PPT / 2];
    float m[PPT];
};

template <int PPT>
__device__ __forceinline__ void fps_load_points(const float *x, int lo, int hi,
                                                int T, ThreadPoints<PPT> &pt,
                                                float *scoord) {
#pragma unroll
    for (int p = 0; p < PPT; ++p) {
        const int j = lo + int(threadIdx.x) + p * T;
        float vx = 0.f, vy = 0.f, vz = 0.f;
        if (j < hi) {
            vx = x[size_t(j) * 3 + 0];
            vy = x[size_t(j) * 3 + 1];
            vz = x[size_t(j) * 3 + 2];
            pt.m[p] = __int_as_float(0x7f800000);  // +inf: first min() gives s
            if (scoord) {
                scoord[(j - lo) * 3 + 0] = vx;
                scoord[(j - lo) * 3 + 1] = vy;
                scoord[(j - lo) * 3 + 2] = vz;
            }
        } else {
            pt.m[p] = -1.0f;  // no point: never the maximum
        }
        if (p & 1) {
            pt.x[p / 2].y = vx;
            pt.y[p / 2].y = vy;
            pt.z[p / 2].y = vz;
        } else {
            pt.x[p / 2].x = vx;
            pt.y[p / 2].x = vy;
            pt.z[p / 2].x = vz;
        }
    }
}

// Steps 1-3: update the owned points with center (cx, cy, cz), reduce the
// block's (key, j) and return it in warp 0's lanes (other warps: undefined).
template <int PPT>
__device__ __forceinline__ void fps_local_step(ThreadPoints<PPT> &pt, float cx,
                                               float cy, float cz, float2 nz0,
                                               int j_first, int T,
                                               uint2 *wslot, unsigned &bhi,
                                               unsigned &bj) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float2 ncx = make_float2(-cx, -cx);
    const float2 ncy = make_float2(-cy, -cy);
    const float2 ncz = make_float2(-cz, -cz);
    float best = -1.0f;
    int bp = 0;
#pragma unroll
    for (int i = 0; i < PPT / 2; ++i) {
        const float2 s = sqdist2(pt.x[i], pt.y[i], pt.z[i], ncx, ncy, ncz, nz0);
        pt.m[2 * i] = fminf(pt.m[2 * i], s.x);
        pt.m[2 * i + 1] = fminf(pt.m[2 * i + 1], s.y);
        if (pt.m[2 * i] > best) {
            best = pt.m[2 * i];
            bp = 2 * i;
        }
        if (pt.m[2 * i + 1] > best) {
            best = pt.m[2 * i + 1];
            bp = 2 * i + 1;
        }
    }
    const unsigned khi = best >= 0.0f ? __float_as_uint(best) + 1u : 0u;
    const unsigned kj = khi ? unsigned(j_first + bp * T) : FULL;
    unsigned whi, wj;
    warp_argmax_hi_min_lo(khi, kj, whi, wj);
    if (lane == 0) wslot[warp] = make_uint2(whi, wj);
    __syncthreads();
    if (warp == 0) {
        const uint2 v = lane < (T >> 5) ? wslot[lane] : make_uint2(0u, FULL);
        warp_argmax_hi_min_lo(v.x, v.y, bhi, bj);
    }
}

// BLOCK (CLUSTER == false, one block per cloud) and CLUSTER schedules.
template <int PPT, bool CLUSTER>
__global__ void __launch_bounds__(fps_max_threads(PPT), 1)
    fps_cluster_kernel(const FpsArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    float *scoord = reinterpret_cast<float *>(smem);
    uint2 *wslot = reinterpret_cast<uint2 *>(smem + fps_coords_bytes(a.chunk));
    ClusterSlot *cslot = reinterpret_cast<ClusterSlot *>(
        smem + fps_coords_bytes(a.chunk) + 32 * sizeof(uint2));
    uint64_t *xbar = reinterpret_cast<uint64_t *>(cslot + 2 * FPS_MAX_CLUSTER);
    int *s_fail = reinterpret_cast<int *>(xbar + 2);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = blockDim.x;
    // CLUSTER: every distributed-shared-memory address below targets ranks
    // < a.nblocks; a launch without that cluster shape stops here (uniform)
    if (CLUSTER && cluster_nctarank() != unsigned(a.nblocks)) {
        if (threadIdx.x == 0) raise_status(a.status, 3 /* PC_ERR_CUDA */);
        return;
    }
    const unsigned rank = CLUSTER ? cluster_ctarank() : 0u;
    const int b = blockIdx.x / a.nblocks;
    const float *x = a.xyz + size_t(b) * size_t(a.N) * 3;
    const int lo = int(rank) * a.chunk;
    const int hi = min(a.N, lo + a.chunk);
    const float2 nz0 = make_float2(a.negzero, a.negzero);
    const unsigned xbytes = unsigned(FPS_CAND_BYTES * a.nblocks);

    ThreadPoints<PPT> pt;
    fps_load_points<PPT>(x, lo, hi, T, pt, scoord);
    float cx = x[size_t(a.start) * 3 + 0];
    float cy = x[size_t(a.start) * 3 + 1];
    float cz = x[size_t(a.start) * 3 + 2];
    int64_t *out = a.out + size_t(b) * a.npoint;
    if (rank == 0 && threadIdx.x == 0) out[0] = a.start;
    if (CLUSTER && threadIdx.x == 0) {
        // one exchange mbarrier per step parity, armed for its first step
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        *s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(&xbar[0], xbytes);
        mbar_arrive_expect_tx(&xbar[1], xbytes);
    }
    __syncthreads();
    if (CLUSTER) cluster_sync_all();  // every block's barriers exist before use

    for (int t = 1; t < a.npoint; ++t) {
        const int par = t & 1;
        unsigned bhi, bj;
        fps_local_step<PPT>(pt, cx, cy, cz, nz0, lo + int(threadIdx.x), T,
                            wslot, bhi, bj);
        if (warp == 0) {
            float wx = 0.f, wy = 0.f, wz = 0.f;
            if (bhi) {
                const float *c = scoord + (int(bj) - lo) * 3;
                wx = c[0];
                wy = c[1];
                wz = c[2];
            }
            ClusterSlot *mine = &cslot[par * FPS_MAX_CLUSTER + rank];
            if (CLUSTER) {
                // testing hook: block 0 of the first cloud withholds step 1
                const bool withhold = (a.stall & 2) && b == 0 && rank == 0 && t == 1;
                if (lane < a.nblocks && !withhold) {
                    const uint32_t ra = map_shared_rank(mine, unsigned(lane));
                    const uint32_t rb = map_shared_rank(&xbar[par], unsigned(lane));
                    st_async_v4(ra, bhi, bj, __float_as_uint(wx),
                                __float_as_uint(wy), rb);
                    st_async_b32(ra + 16, __float_as_uint(wz), rb);
                }
            } else if (lane == 0) {
                mine->hi = bhi;
                mine->j = bj;
                mine->x = wx;
                mine->y = wy;
                mine->z = wz;
            }
        }
        if (CLUSTER) {
            const unsigned ph = unsigned((t - 1) >> 1) & 1u;
            const bool got = mbar_wait_cluster_bounded(&xbar[par], ph, a.timeout_ns);
            if (!got) *s_fail = 1;
            // re-arm this parity's barrier for step t + 2 (its next phase
            // cannot complete before every block has passed this point);
            // only after seeing this phase complete: a phase that ran out
            // still holds its arrival, and the kernel stops anyway
            if (threadIdx.x == 0 && got) mbar_arrive_expect_tx(&xbar[par], xbytes);
            if (__syncthreads_or(*s_fail)) {
                raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
                if (rank == 0)
                    for (int i = t + int(threadIdx.x); i < a.npoint; i += T)
                        out[i] = -1;
                break;
            }
        } else {
            __syncthreads();
        }
        // every warp reduces the cloud's candidates
        const ClusterSlot *cs = &cslot[par * FPS_MAX_CLUSTER];
        unsigned vhi = 0u, vj = FULL;
        float vx = 0.f, vy = 0.f, vz = 0.f;
        if (lane < a.nblocks) {
            vhi = cs[lane].hi;
            vj = cs[lane].j;
            vx = cs[lane].x;
            vy = cs[lane].y;
            vz = cs[lane].z;
        }
        unsigned chi, cj;
        warp_argmax_hi_min_lo(vhi, vj, chi, cj);
        const int who = __ffs(__ballot_sync(FULL, vhi == chi && vj == cj)) - 1;
        cx = __shfl_sync(FULL, vx, who);
        cy = __shfl_sync(FULL, vy, who);
        cz = __shfl_sync(FULL, vz, who);
        if (rank == 0 && threadIdx.x == 0) out[t] = int64_t(cj);
    }
    if (CLUSTER) cluster_sync_all();  // no block exits while peers may write
}

// ---------------------------------------------------------------------------
// CLUSTER schedule in rounds: several centers per exchange.
//
// The sequential rule takes, at every step, the point of largest m (smallest
// index on a tie).  A round certifies a run of such steps from a short list:
//   * every warp lists its own best point (largest m, smallest index) and up
//     to FR_CW - 1 more lane-best points, and bounds every point it does not
//     list: a point that is not its lane's best is at most the lane's second
//     largest m, and a lane-best point that is not listed is at most the
//     warp's bound by construction (lanes whose best exceeds the bound are
//     listed, those past FR_CW raise the bound to their m);
//   * the blocks of the cloud exchange their lists and bounds (one bulk copy
//     into every block's shared memory), and every block resolves the same
//     run: the first center is the largest listed point -- the cloud's
//     largest, since every warp's best is listed; after it the listed points'
//     m are lowered by the new center exactly as the step would lower them,
//     and the next largest listed point is the next center as long as its m
//     is strictly above B, the largest bound, which every unlisted point's m
//     stays at or below.  The run ends at the first point that is not above
//     B (or after FR_RMAX centers);
//   * every block then lowers its points' m by the run's centers (min is
//     exact in any order) and lists again.
// Each accepted center is the one the step-by-step rule takes, so the
// output is identical; a round costs one exchange for the whole run (100k
// points, 4096 samples: about 27 centers a round).
//
// A block has one more warp than it needs for its points: that warp holds
// none; it sends the block's list, and after the scan (every warp's share)
// it certifies the run and publishes each center in shared memory as it is
// taken, while the point warps lower their m by the published centers -- the
// sequential picks overlap the point work (GB300, 100k points on 13 blocks:
// 2.56 ms with warp 0 picking and updating its own points afterwards, 2.20
// with the extra warp).
constexpr int FR_CW = 8;     // entries a warp lists per round (its best first)
constexpr int FR_RMAX = 64;  // centers a round takes at most
constexpr int FR_LIST = 4;   // certified candidates a lane of the resolving warp holds

// A listed point: key (bits(m) + 1; 0 = empty), original index, coordinates.
struct __align__(16) FrEntry {
    unsigned hi, j;
    float x, y;
    float z, pad0, pad1, pad2;
};

// A block's list: [W warps][FR_CW] entries, then [W] bounds (uint4: key, -).
__host__ __device__ constexpr unsigned fr_msg_bytes(int warps) {
    return unsigned(warps) * FR_CW * 32u + unsigned(warps) * 16u;
}

__host__ __device__ constexpr size_t fr_align16(size_t v) { return (v + 15) & ~size_t(15); }

// Shared memory: the block's points (12 B each), its list, the lists of the
// cloud's blocks by round parity, the run's centers, the candidate
// offsets, each warp's largest entry, the lists' counts of candidates, the
// exchange mbarriers and six counters/flags.
__host__ __device__ constexpr size_t fps_rounds_smem(int chunk, int warps, int nblocks) {
    return fr_align16(size_t(chunk) * 12) + fr_msg_bytes(warps) +
           2 * size_t(nblocks) * fr_msg_bytes(warps) +
           size_t(FR_RMAX) * 16 + 32 * FR_LIST * sizeof(int) + 32 * sizeof(uint4) +
           FPS_MAX_CLUSTER * sizeof(int) + 2 * sizeof(uint64_t) + 32;
}

// Every warp of a block (nscan of them), once the round's lists are in,
// pass 1: B, the largest bound of an unlisted point (returned); for lists
// warp, warp + nscan, ... the number of entries above B (cnt[list]) and the
// warp's largest entry (smallest index on a tie) in *wfirst as (key, index,
// offset).  A list is `msg` bytes: `per` entries, then `nbnd` bounds (uint4,
// key in .x) -- a block's list (per = W * FR_CW, nbnd = W) or a cluster's
// summary (per = FR_SUM, nbnd = 1), of which only the first lens[l] entries
// are read when lens is given.
__device__ __forceinline__ unsigned fr_count(const unsigned char *lists, int nl, int per,
                                             int nbnd, int nscan, unsigned msg, int *cnt,
                                             uint4 *wfirst, const int *lens = nullptr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the bounds: lane = (list of its group, bound), 32 / nbnd lists at a time
    unsigned bnd = 0u;
    const int lpi = 32 / nbnd, li = lane / nbnd, bi = lane - li * nbnd;
    if (li < lpi)
        for (int l = li; l < nl; l += lpi)
            bnd = max(bnd, reinterpret_cast<const uint4 *>(lists + size_t(l) * msg +
                                                           size_t(per) * 32)[bi].x);
    bnd = __reduce_max_sync(FULL, bnd);
    unsigned gh = 0u, gj = FULL;
    int go = 0;
    for (int l = warp; l < nl; l += nscan) {
        int n = 0;
        const int len = lens ? lens[l] : per;
        for (int k0 = 0; k0 < len; k0 += 32) {
            const int k = k0 + lane;
            const int off = l * int(msg) + k * 32;
            unsigned h = 0u, j = FULL;
            if (k < len) {
                const uint2 hj = *reinterpret_cast<const uint2 *>(lists + off);
                h = hj.x;
                j = hj.y;
            }
            if (h > gh || (h == gh && h != 0u && j < gj)) {
                gh = h;
                gj = j;
                go = off;
            }
            n += __popc(__ballot_sync(FULL, h > bnd));
        }
        if (lane == 0) cnt[l] = n;
    }
    unsigned wh, wj;
    warp_argmax_hi_min_lo(gh, gj, wh, wj);
    const unsigned holder = __ballot_sync(FULL, gh == wh && gj == wj);
    if (lane == __ffs(holder) - 1) *wfirst = make_uint4(wh, wj, unsigned(go), 0u);
    return bnd;
}

// The sum of cnt[0 .. l) (l <= nl, the same in every lane of the warp).
__device__ __forceinline__ int fr_before(const int *cnt, int l) {
    const int lane = threadIdx.x & 31;
    int acc = 0;
    for (int i = lane; i < l; i += 32) acc += cnt[i];
    return __reduce_add_sync(FULL, acc);
}

// Pass 2, after a barrier: every entry above B gets the candidate position
// 1 + (entries above B in the lists before its own) + (those before it in its
// list) -- the same in every block of the cloud, whatever the warps' timing
// -- and its byte offset goes to cidx; the ones at positions past
// 32 * FR_LIST raise *s_over to their m instead (every block then keeps the
// same candidates and the same bound, and certifies the same run).
__device__ __forceinline__ void fr_place(const unsigned char *lists, int nl, int per,
                                         int nscan, unsigned msg, unsigned bnd,
                                         const int *cnt, int *cidx, unsigned *s_over,
                                         const int *lens = nullptr) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int CAP = 32 * FR_LIST;
    unsigned over = 0u;
    for (int l = warp; l < nl; l += nscan) {
        int base = 1 + fr_before(cnt, l);
        const int len = lens ? lens[l] : per;
        for (int k0 = 0; k0 < len; k0 += 32) {
            const int k = k0 + lane;
            const int off = l * int(msg) + k * 32;
            const unsigned h = k < len ? *reinterpret_cast<const unsigned *>(lists + off) : 0u;
            const bool keep = h > bnd;
            const unsigned bal = __ballot_sync(FULL, keep);
            const int pos = base + __popc(bal & lanemask_lt());
            if (keep) {
                if (pos < CAP)
                    cidx[pos] = off;
                else
                    over = max(over, h);
            }
            base += __popc(bal);
        }
    }
    over = __reduce_max_sync(FULL, over);
    if (lane == 0 && over != 0u) atomicMax(s_over, over);
}

// The resolving warp of a block, after fr_count and fr_place:
// the run of centers the lists certify (see above).  Writes the centers to
// cen[0 .. k), publishing each in *s_pub as it is taken (the point warps
// apply it meanwhile), their indices to out[0 .. k) when out is given, k to
// *s_nc, and sets *s_fin at the end.
__device__ __forceinline__ void fr_pick(const unsigned char *lists, int nscan, unsigned bnd,
                                        int rmax, const int *cidx, const uint4 *wfirst,
                                        int total, unsigned over, float4 *cen, int *s_nc,
                                        volatile int *s_pub, volatile int *s_fin,
                                        int64_t *out) {
    const int lane = threadIdx.x & 31;
    constexpr int CAP = 32 * FR_LIST;
    bnd = max(bnd, over);
    // the first center: the largest of the warps' largest entries
    const uint4 f = lane < nscan ? wfirst[lane] : make_uint4(0u, FULL, 0u, 0u);
    unsigned fh, fj;
    warp_argmax_hi_min_lo(f.x, f.y, fh, fj);
    if (fh == 0u) {  // no point at all (cannot happen for N >= 1): stop the run
        if (lane == 0) {
            *s_nc = 0;
            __threadfence_block();
            *s_fin = 1;
        }
        return;
    }
    const int first = int(__shfl_sync(
        FULL, f.z, __ffs(__ballot_sync(FULL, f.x == fh && f.y == fj)) - 1));
    const int nlist = min(total, CAP);
    unsigned lh[FR_LIST], lj[FR_LIST];
    float lx[FR_LIST], ly[FR_LIST], lz[FR_LIST];
#pragma unroll
    for (int s = 0; s < FR_LIST; ++s) {
        const int q = lane + 32 * s;
        const int off = q == 0 ? first : (q < nlist ? cidx[q] : -1);
        lh[s] = 0u;
        lj[s] = FULL;
        lx[s] = ly[s] = lz[s] = 0.f;
        if (off >= 0 && (q == 0 || off != first)) {  // the first center also above B: once
            const FrEntry *e = reinterpret_cast<const FrEntry *>(lists + off);
            lh[s] = e->hi;
            lj[s] = e->j;
            lx[s] = e->x;
            ly[s] = e->y;
            lz[s] = e->z;
        }
    }
    int k = 0;
    for (; k < rmax; ++k) {
        // the lane's largest candidate (smallest index on a tie): slots 0-1
        // and 2-3, then the two winners
        static_assert(FR_LIST == 4, "the pairwise choice below takes four slots");
        const bool r01 = lh[1] > lh[0] || (lh[1] == lh[0] && lj[1] < lj[0]);
        const bool r23 = lh[3] > lh[2] || (lh[3] == lh[2] && lj[3] < lj[2]);
        const unsigned ha = r01 ? lh[1] : lh[0], ja = r01 ? lj[1] : lj[0];
        const unsigned hb = r23 ? lh[3] : lh[2], jb = r23 ? lj[3] : lj[2];
        const bool rab = hb > ha || (hb == ha && jb < ja);
        const unsigned bh = rab ? hb : ha, bj = rab ? jb : ja;
        const unsigned wh = __reduce_max_sync(FULL, bh);
        // the first center is the cloud's largest; a later one must be above
        // every unlisted point's m
        if (wh == 0u || (k > 0 && wh <= bnd)) break;
        unsigned top = __ballot_sync(FULL, bh == wh);
        if (__popc(top) > 1) {  // equal m in several lanes: the smallest index
            const unsigned wj = __reduce_min_sync(FULL, bh == wh ? bj : FULL);
            top = __ballot_sync(FULL, bh == wh && bj == wj);
        }
        const int wl = __ffs(top) - 1;
        const float xa = r01 ? lx[1] : lx[0], ya = r01 ? ly[1] : ly[0], za = r01 ? lz[1] : lz[0];
        const float xb = r23 ? lx[3] : lx[2], yb = r23 ? ly[3] : ly[2], zb = r23 ? lz[3] : lz[2];
        const float cx = __shfl_sync(FULL, rab ? xb : xa, wl);
        const float cy = __shfl_sync(FULL, rab ? yb : ya, wl);
        const float cz = __shfl_sync(FULL, rab ? zb : za, wl);
        const unsigned cj = __shfl_sync(FULL, bj, wl);
        if (lane == 0) {  // the center (its index in .w), then its publication
            cen[k] = make_float4(cx, cy, cz, __uint_as_float(cj));
            __threadfence_block();
            *s_pub = k + 1;
        }
        // lower the candidates' m by the new center, as the step would (a
        // NaN distance leaves m, as fminf does)
#pragma unroll
        for (int s = 0; s < FR_LIST; ++s) {
            const float sv = sqdist(lx[s], ly[s], lz[s], cx, cy, cz);
            const unsigned kv = sv >= 0.0f ? __float_as_uint(sv) + 1u : FULL;
            lh[s] = lh[s] != 0u ? min(lh[s], kv) : 0u;
        }
    }
    if (lane == 0) {
        *s_nc = k;
        __threadfence_block();
        *s_fin = 1;
    }
    // the run's indices, after the run: a global store inside the loop would
    // hold up the next center's fence until it completed
    if (out) {
        __syncwarp();
        for (int i = lane; i < k; i += 32) out[i] = int64_t(__float_as_uint(cen[i].w));
    }
}

// A point warp's list for the round (every lane of the warp): its entries
// at mine[0 .. FR_CW) (empty ones with key 0) and its bound at *mybound.
template <int PPT>
__device__ __forceinline__ void fr_list(const ThreadPoints<PPT> &pt, const float *scoord,
                                        int lo, int T, FrEntry *mine, uint4 *mybound) {
    const int lane = threadIdx.x & 31;
    // the lane's best point (its slots are in increasing index, so a
    // strict ">" keeps the smaller index on a tie) and its second largest m
    float best = -1.0f, second = -1.0f;
    int bp = 0;
#pragma unroll
    for (int p = 0; p < PPT; ++p) {
        const float v = pt.m[p];
        if (v > best) {
            second = best;
            best = v;
            bp = p;
        } else {
            second = fmaxf(second, v);
        }
    }
    const unsigned khi = best >= 0.0f ? __float_as_uint(best) + 1u : 0u;
    const unsigned kj = khi ? unsigned(lo + bp * T + int(threadIdx.x)) : FULL;
    const unsigned shi = second >= 0.0f ? __float_as_uint(second) + 1u : 0u;
    // the warp's list (its best first, then lanes whose best is above
    // the bound, in lane order) and its bound
    unsigned whi, wj;
    warp_argmax_hi_min_lo(khi, kj, whi, wj);
    const int wl = __ffs(__ballot_sync(FULL, khi == whi && kj == wj)) - 1;
    unsigned bw = __reduce_max_sync(FULL, shi);
    const unsigned cand = __ballot_sync(FULL, khi > bw && lane != wl);
    const int crank = __popc(cand & lanemask_lt());
    const bool is_c = (cand >> lane) & 1u;
    bw = max(bw, __reduce_max_sync(FULL, is_c && crank >= FR_CW - 1 ? khi : 0u));
    const bool listed = (lane == wl && whi != 0u) || (is_c && crank < FR_CW - 1);
    if (listed) {
        const float *c = scoord + (int(kj) - lo) * 3;
        FrEntry *e = mine + (lane == wl ? 0 : 1 + crank);
        e->hi = khi;
        e->j = kj;
        e->x = c[0];
        e->y = c[1];
        e->z = c[2];
    }
    const int nlisted = (whi != 0u ? 1 : 0) + min(__popc(cand), FR_CW - 1);
    if (lane >= nlisted && lane < FR_CW) mine[lane].hi = 0u;
    if (lane == 0) *mybound = make_uint4(bw, 0u, 0u, 0u);
}

// Threads a rounds kernel with PPT points per thread may use: the point
// threads of the schedules (at most 256 with 32 points, 384 with fewer) and
// the resolving warp.
__host__ __device__ constexpr int fr_max_threads(int ppt) { return ppt >= 32 ? 288 : 416; }

template <int PPT>
__global__ void __launch_bounds__(fr_max_threads(PPT), 1)
    fps_rounds_kernel(const FpsArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = int(blockDim.x) - 32;  // threads holding points
    const int W = T >> 5;                // their warps, which list
    const int NW = W + 1;                // and the resolving warp
    const bool rw = warp == W;
    const unsigned msg = fr_msg_bytes(W);
    float *scoord = reinterpret_cast<float *>(smem);
    unsigned char *sbuf = smem + fr_align16(size_t(a.chunk) * 12);
    unsigned char *recv = sbuf + msg;  // [2 parities][nblocks] lists
    float4 *cen = reinterpret_cast<float4 *>(recv + 2 * size_t(a.nblocks) * msg);
    int *cidx = reinterpret_cast<int *>(cen + FR_RMAX);
    uint4 *wfirst = reinterpret_cast<uint4 *>(cidx + 32 * FR_LIST);
    int *lcnt = reinterpret_cast<int *>(wfirst + 32);  // [nblocks] candidates per list
    uint64_t *xbar = reinterpret_cast<uint64_t *>(lcnt + FPS_MAX_CLUSTER);
    int *s_nc = reinterpret_cast<int *>(xbar + 2);
    int *s_fail = s_nc + 1;
    int *s_total = s_nc + 2;  // candidate positions taken (position 0: the first center)
    unsigned *s_over = reinterpret_cast<unsigned *>(s_nc + 3);
    volatile int *s_pub = s_nc + 4;  // centers of the run published so far
    volatile int *s_fin = s_nc + 5;  // the run is complete

    // every distributed-shared-memory address below targets ranks
    // < a.nblocks; a launch without that cluster shape stops here (uniform)
    if (cluster_nctarank() != unsigned(a.nblocks)) {
        if (threadIdx.x == 0) raise_status(a.status, 3 /* PC_ERR_CUDA */);
        return;
    }
    const unsigned rank = cluster_ctarank();
    const int b = blockIdx.x / a.nblocks;
    const float *x = a.xyz + size_t(b) * size_t(a.N) * 3;
    const int lo = int(rank) * a.chunk;
    const int hi = min(a.N, lo + a.chunk);
    const float2 nz0 = make_float2(a.negzero, a.negzero);
    const unsigned xbytes = unsigned(a.nblocks) * msg;

    ThreadPoints<PPT> pt;
    if (!rw) {
        fps_load_points<PPT>(x, lo, hi, T, pt, scoord);
    } else {
#pragma unroll
        for (int p = 0; p < PPT; ++p) pt.m[p] = -1.0f;
#pragma unroll
        for (int i = 0; i < PPT / 2; ++i) pt.x[i] = pt.y[i] = pt.z[i] = make_float2(0.f, 0.f);
    }
    int64_t *out = a.out + size_t(b) * a.npoint;
    if (threadIdx.x == 0) {
        cen[0] = make_float4(x[size_t(a.start) * 3 + 0], x[size_t(a.start) * 3 + 1],
                             x[size_t(a.start) * 3 + 2], 0.f);
        *s_nc = 1;
        *s_fail = 0;
        *s_total = 1;
        *s_over = 0u;
        *s_pub = 0;
        *s_fin = 0;
        if (rank == 0) out[0] = a.start;
        // one exchange mbarrier per round parity, armed for its first round
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(&xbar[0], xbytes);
        mbar_arrive_expect_tx(&xbar[1], xbytes);
    }
    __syncthreads();
    cluster_sync_all();  // every block's barriers exist before use

    // lower the thread's points' m by the center cc
    auto apply = [&](const float4 cc) {
        const float2 ncx = make_float2(-cc.x, -cc.x);
        const float2 ncy = make_float2(-cc.y, -cc.y);
        const float2 ncz = make_float2(-cc.z, -cc.z);
#pragma unroll
        for (int i = 0; i < PPT / 2; ++i) {
            const float2 s = sqdist2(pt.x[i], pt.y[i], pt.z[i], ncx, ncy, ncz, nz0);
            pt.m[2 * i] = fminf(pt.m[2 * i], s.x);
            pt.m[2 * i + 1] = fminf(pt.m[2 * i + 1], s.y);
        }
    };
    // lower them by two centers at once (min is exact in any order)
    auto apply2 = [&](const float4 c0, const float4 c1) {
        const float2 ncx = make_float2(-c0.x, -c0.x);
        const float2 ncy = make_float2(-c0.y, -c0.y);
        const float2 ncz = make_float2(-c0.z, -c0.z);
        const float2 mcx = make_float2(-c1.x, -c1.x);
        const float2 mcy = make_float2(-c1.y, -c1.y);
        const float2 mcz = make_float2(-c1.z, -c1.z);
#pragma unroll
        for (int i = 0; i < PPT / 2; ++i) {
            const float2 s = sqdist2(pt.x[i], pt.y[i], pt.z[i], ncx, ncy, ncz, nz0);
            const float2 u = sqdist2(pt.x[i], pt.y[i], pt.z[i], mcx, mcy, mcz, nz0);
            pt.m[2 * i] = fmin3(pt.m[2 * i], s.x, u.x);
            pt.m[2 * i + 1] = fmin3(pt.m[2 * i + 1], s.y, u.y);
        }
    };
    FrEntry *mine = reinterpret_cast<FrEntry *>(sbuf) + warp * FR_CW;
    uint4 *mybound = reinterpret_cast<uint4 *>(sbuf + size_t(W) * FR_CW * 32) + warp;
    int t = 1;  // centers output so far
    for (int round = 0; t < a.npoint; ++round) {
        const int par = round & 1;
        // 1. the start lowers the points' m (later centers were applied while
        // the resolving warp picked them)
        if (round == 0 && !rw) apply(cen[0]);
        if (!rw) fr_list<PPT>(pt, scoord, lo, T, mine, mybound);
        fence_proxy_async_smem();  // the list, for the bulk copies
        __syncthreads();
        if (rw) {
            // testing hook: block 0 of the first cloud withholds round 0
            const bool withhold = (a.stall & 2) && b == 0 && rank == 0 && round == 0;
            if (lane < a.nblocks && !withhold) {
                const uint32_t dst = map_shared_rank(
                    recv + (size_t(par) * a.nblocks + rank) * msg, unsigned(lane));
                const uint32_t bar = map_shared_rank(&xbar[par], unsigned(lane));
                bulk_copy_to_cluster(dst, sbuf, msg, bar);
                bulk_commit();
            }
        }
        // 4. the round's lists are in: every warp waits (bounded); thread 0
        // re-arms this parity for round + 2 (its next phase cannot complete
        // before every block has passed this round)
        {
            const unsigned ph = unsigned(round >> 1) & 1u;
            const bool got =
                __all_sync(FULL, mbar_wait_cluster_bounded(&xbar[par], ph, a.timeout_ns));
            if (threadIdx.x == 0 && got) mbar_arrive_expect_tx(&xbar[par], xbytes);
            // the list may be rewritten once this round is over
            if (rw && lane < a.nblocks) bulk_wait_read_all();
            if (!got && lane == 0) *s_fail = 1;
        }
        // 5. every warp scans its share of the lists; the resolving warp
        // certifies the run
        const unsigned char *lists = recv + size_t(par) * a.nblocks * msg;
        const unsigned bnd =
            fr_count(lists, a.nblocks, W * FR_CW, W, NW, msg, lcnt, wfirst + warp);
        __syncthreads();
        fr_place(lists, a.nblocks, W * FR_CW, NW, msg, bnd, lcnt, cidx, s_over);
        if (warp == 0) {  // candidates in all: the first center and the counts
            const int total = 1 + fr_before(lcnt, a.nblocks);
            if (lane == 0) *s_total = total;
        }
        __syncthreads();
        if (rw) {
            if (!*s_fail)
                fr_pick(lists, NW, bnd, min(FR_RMAX, a.npoint - t), cidx, wfirst, *s_total,
                        *s_over, cen, s_nc, s_pub, s_fin, rank == 0 ? out + t : nullptr);
            else if (lane == 0)
                *s_fin = 1;
        } else {
            // apply the run's centers as the resolving warp publishes them
            // (bounded wait: the run is short, the limit is a safety net)
            // (a warp that finds nothing new sleeps briefly instead of polling:
            // its loads and fences would slow the resolving warp's shuffles)
            int c = 0;
            const uint64_t w0 = global_timer_ns();
            for (int spin = 0;; ++spin) {
                const int fin = *s_fin;
                const int pub = *s_pub;
                if (pub > c || fin) {
                    __threadfence_block();  // the centers published before pub / fin
                    const int upto = fin ? *s_pub : pub;
                    while (c < upto) {  // two at a time where two are out
                        if (c + 1 < upto) {
                            apply2(cen[c], cen[c + 1]);
                            c += 2;
                        } else {
                            apply(cen[c]);
                            ++c;
                        }
                    }
                    if (fin) break;
                    continue;
                }
                __nanosleep(32);
                if ((spin & 63) == 63 && global_timer_ns() - w0 > a.timeout_ns) {
                    if (lane == 0) *s_fail = 1;
                    break;
                }
            }
        }
        __syncthreads();
        const int taken = *s_nc;
        if (*s_fail || taken <= 0) {
            raise_status(a.status, *s_fail ? 4 /* PC_ERR_DEVICE_TIMEOUT */ : 3 /* PC_ERR_CUDA */);
            if (rank == 0)
                for (int i = t + int(threadIdx.x); i < a.npoint; i += T) out[i] = -1;
            break;
        }
        t += taken;
        if (threadIdx.x == 0) {  // for the next round
            *s_total = 1;
            *s_over = 0u;
            *s_pub = 0;
            *s_fin = 0;
        }
    }
    // no copy in flight and no block exits while peers may write
    if (rw && lane < a.nblocks) bulk_wait_all();
    cluster_sync_all();
}

// GRID schedule: cooperative launch, a.nblocks blocks per cloud.
template <int PPT>
__global__ void __launch_bounds__(fps_max_threads(PPT), 1)
    fps_grid_kernel(const FpsArgs a) {
    __shared__ uint2 wslot[32];
    __shared__ float4 s_center;
    __shared__ int s_fail;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = blockDim.x;
    const int b = blockIdx.x / a.nblocks;
    const int r = blockIdx.x % a.nblocks;
    const float *x = a.xyz + size_t(b) * size_t(a.N) * 3;
    const int lo = r * a.chunk;
    const int hi = min(a.N, lo + a.chunk);
    uint64_t *slots = a.slots + size_t(b) * 2 * a.nblocks;
    const float2 nz0 = make_float2(a.negzero, a.negzero);

    ThreadPoints<PPT> pt;
    fps_load_points<PPT>(x, lo, hi, T, pt, nullptr);
    float cx = x[size_t(a.start) * 3 + 0];
    float cy = x[size_t(a.start) * 3 + 1];
    float cz = x[size_t(a.start) * 3 + 2];
    int64_t *out = a.out + size_t(b) * a.npoint;
    if (r == 0 && threadIdx.x == 0) out[0] = a.start;
    if (threadIdx.x == 0) s_fail = 0;

    int t = 1;
    for (; t < a.npoint; ++t) {
        const int par = t & 1;
        const unsigned tag = unsigned(t) & 511u;
        unsigned bhi, bj;
        fps_local_step<PPT>(pt, cx, cy, cz, nz0, lo + int(threadIdx.x), T,
                            wslot, bhi, bj);
        if (warp == 0) {
            uint64_t *ps = slots + size_t(par) * a.nblocks;
            if (lane == 0 && !((a.stall & 1) && r == 0 && t == 1)) {
                const uint64_t key =
                    (uint64_t(bhi) << 33) |
                    (uint64_t((FPS_GRID_MAX_N - 1) - (bhi ? bj : 0u)) << 9) |
                    tag;
                st_relaxed_gpu_u64(&ps[r], key);
            }
            // poll until every block of the cloud published this step
            uint64_t best = 0;
            bool ok = false;
            const uint64_t t0 = global_timer_ns();
            for (int spin = 0;; ++spin) {
                bool mine_ok = true;
                uint64_t m = 0;
                for (int i = lane; i < a.nblocks; i += 32) {
                    const uint64_t v = ld_relaxed_gpu_u64(&ps[i]);
                    if ((v & 511u) != tag)
                        mine_ok = false;
                    else
                        m = v > m ? v : m;
                }
                if (__all_sync(FULL, mine_ok)) {
                    best = m;
                    ok = true;
                    break;
                }
                if ((spin & 63) == 63 &&
                    global_timer_ns() - t0 > a.timeout_ns)
                    break;
            }
            if (!ok) {
                if (lane == 0) {
                    s_fail = 1;
                    raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
                }
            } else {
                const unsigned mhi = __reduce_max_sync(FULL, unsigned(best >> 32));
                const unsigned lo32 = __reduce_max_sync(
                    FULL, unsigned(best >> 32) == mhi ? unsigned(best) : 0u);
                const uint64_t w = (uint64_t(mhi) << 32) | lo32;
                const unsigned wj =
                    (FPS_GRID_MAX_N - 1) - unsigned((w >> 9) & 0xffffffu);
                if (lane == 0) {
                    s_center = make_float4(x[size_t(wj) * 3 + 0],
                                           x[size_t(wj) * 3 + 1],
                                           x[size_t(wj) * 3 + 2],
                                           __int_as_float(int(wj)));
                    if (r == 0) out[t] = int64_t(wj);
                }
            }
        }
        __syncthreads();
        if (s_fail) break;
        const float4 c = s_center;
        cx = c.x;
        cy = c.y;
        cz = c.z;
    }
    if (s_fail && r == 0) {
        for (int i = t + int(threadIdx.x); i < a.npoint; i += T) out[i] = -1;
    }
}

// GRID schedule in two levels: a cooperative launch of thread block
// clusters of a.cs blocks, a.ncl clusters (a.nblocks = a.cs * a.ncl blocks)
// per cloud.  Per step:
//   1. every block of a cluster sends its candidate (key, coordinates) to
//      the cluster's block 0 (its leader) through distributed shared memory
//      with st.async, and the leader reduces them to the cluster's best;
//   2. block 0 of each cluster (its leader) publishes that best into the
//      cluster's slot of the workspace -- four 64-bit words on a 128-byte
//      line of their own, each carrying the step's tag in its low 9 bits:
//          key  [bits(m)+1 : 31 | 2^24-1-j : 24 | step mod 512 : 9]
//          x, y, z  [float bits : 32 | 0 : 23 | step mod 512 : 9]
//      -- and polls the cloud's a.ncl slots until every word carries this
//      step's tag (each word is checked on its own, so the stores need no
//      ordering, and the winner's coordinates arrive with its key);
//   3. the leader sends the winner to every block of its cluster through
//      distributed shared memory (st.async on a second mbarrier pair).
// Only the a.ncl leaders touch the workspace, so a step's global exchange is
// a.ncl writers and a.ncl readers of a.ncl lines (GB300, 1M points, 16,384
// samples: 31.7 ms with every block's candidate sent to every block of its
// cluster, 30.9 ms with it sent to the leader only).  Double buffering by step
// parity holds at every level: a block sends step t + 2 only after its
// leader read every cluster's step t + 1, which each cluster publishes only
// after all its blocks finished step t.  Every wait is bounded.
template <int PPT>
__global__ void __launch_bounds__(fps_max_threads(PPT), 1)
    fps_cgrid_kernel(const FpsArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    float *scoord = reinterpret_cast<float *>(smem);
    uint2 *wslot = reinterpret_cast<uint2 *>(smem + fps_coords_bytes(a.chunk));
    ClusterSlot *cslot = reinterpret_cast<ClusterSlot *>(
        smem + fps_coords_bytes(a.chunk) + 32 * sizeof(uint2));
    uint64_t *xbar = reinterpret_cast<uint64_t *>(cslot + 2 * FPS_MAX_CLUSTER);
    int *s_fail = reinterpret_cast<int *>(xbar + 2);
    uint64_t *bbar = xbar + 4;                                   // [2]
    ClusterSlot *bslot = reinterpret_cast<ClusterSlot *>(xbar + 6);  // [2]

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = blockDim.x;
    // every distributed-shared-memory address below targets ranks < a.cs:
    // a launch without that cluster shape stops here, before any access
    // (uniform over the launch, so no block is left waiting)
    if (cluster_nctarank() != unsigned(a.cs)) {
        if (threadIdx.x == 0) raise_status(a.status, 3 /* PC_ERR_CUDA */);
        return;
    }
    const unsigned rank = cluster_ctarank();
    const int b = blockIdx.x / a.nblocks;
    const int r = blockIdx.x % a.nblocks;  // block of the cloud
    const int cl = r / a.cs;               // cluster of the cloud
    const float *x = a.xyz + size_t(b) * size_t(a.N) * 3;
    const int lo = r * a.chunk;
    const int hi = min(a.N, lo + a.chunk);
    // slot i of parity p: words [(p * ncl + i) * CG_SLOT_WORDS, + 4)
    uint64_t *slots = a.slots + size_t(b) * 2 * a.ncl * CG_SLOT_WORDS;
    const float2 nz0 = make_float2(a.negzero, a.negzero);
    const unsigned xbytes = unsigned(FPS_CAND_BYTES * a.cs);

    ThreadPoints<PPT> pt;
    fps_load_points<PPT>(x, lo, hi, T, pt, scoord);
    float cx = x[size_t(a.start) * 3 + 0];
    float cy = x[size_t(a.start) * 3 + 1];
    float cz = x[size_t(a.start) * 3 + 2];
    int64_t *out = a.out + size_t(b) * a.npoint;
    if (r == 0 && threadIdx.x == 0) out[0] = a.start;
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&xbar[i], 1);
            mbar_init(&bbar[i], 1);
        }
        *s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int i = 0; i < 2; ++i) {
            mbar_arrive_expect_tx(&xbar[i], xbytes);
            mbar_arrive_expect_tx(&bbar[i], FPS_CAND_BYTES);
        }
    }
    __syncthreads();
    cluster_sync_all();  // every block's barriers exist before use

    bool failed = false;
    int t = 1;
    for (; t < a.npoint; ++t) {
        const int par = t & 1;
        const unsigned tag = unsigned(t) & 511u;
        const unsigned ph = unsigned((t - 1) >> 1) & 1u;
        unsigned bhi, bj;
        fps_local_step<PPT>(pt, cx, cy, cz, nz0, lo + int(threadIdx.x), T,
                            wslot, bhi, bj);
        // 1. the block's candidate to the cluster's leader (rank 0)
        if (warp == 0 && lane == 0) {
            float wx = 0.f, wy = 0.f, wz = 0.f;
            if (bhi) {
                const float *c = scoord + (int(bj) - lo) * 3;
                wx = c[0];
                wy = c[1];
                wz = c[2];
            }
            ClusterSlot *mine = &cslot[par * FPS_MAX_CLUSTER + rank];
            const uint32_t ra = map_shared_rank(mine, 0u);
            const uint32_t rb = map_shared_rank(&xbar[par], 0u);
            st_async_v4(ra, bhi, bj, __float_as_uint(wx), __float_as_uint(wy), rb);
            st_async_b32(ra + 16, __float_as_uint(wz), rb);
        }
        if (rank == 0) {  // the leader: steps 1 to 3
            const bool got = mbar_wait_cluster_bounded(&xbar[par], ph, a.timeout_ns);
            if (threadIdx.x == 0 && got) mbar_arrive_expect_tx(&xbar[par], xbytes);
            if (__syncthreads_or(!got)) {
                if (threadIdx.x == 0) raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
                failed = true;
                break;
            }
            if (warp == 0) {
                const ClusterSlot *cs = &cslot[par * FPS_MAX_CLUSTER];
                unsigned vhi = 0u, vj = FULL;
                float vx = 0.f, vy = 0.f, vz = 0.f;
                if (lane < a.cs) {
                    vhi = cs[lane].hi;
                    vj = cs[lane].j;
                    vx = cs[lane].x;
                    vy = cs[lane].y;
                    vz = cs[lane].z;
                }
                unsigned chi, cj;
                warp_argmax_hi_min_lo(vhi, vj, chi, cj);
                const int who = __ffs(__ballot_sync(FULL, vhi == chi && vj == cj)) - 1;
                const float kx = __shfl_sync(FULL, vx, who);
                const float ky = __shfl_sync(FULL, vy, who);
                const float kz = __shfl_sync(FULL, vz, who);
                uint64_t *gs = slots + size_t(par) * a.ncl * CG_SLOT_WORDS;
                // testing hook: cluster 0 of the first cloud withholds step 1
                const bool withhold = (a.stall & 1) && b == 0 && cl == 0 && t == 1;
                if (lane == 0 && !withhold) {
                    uint64_t *w = gs + size_t(cl) * CG_SLOT_WORDS;
                    st_relaxed_gpu_u64(w + 1, (uint64_t(__float_as_uint(kx)) << 32) | tag);
                    st_relaxed_gpu_u64(w + 2, (uint64_t(__float_as_uint(ky)) << 32) | tag);
                    st_relaxed_gpu_u64(w + 3, (uint64_t(__float_as_uint(kz)) << 32) | tag);
                    st_relaxed_gpu_u64(
                        w, (uint64_t(chi) << 33) |
                               (uint64_t((FPS_GRID_MAX_N - 1) - (chi ? cj : 0u)) << 9) | tag);
                }
                uint64_t mk = 0;
                float mx = 0.f, my = 0.f, mz = 0.f;
                bool ok = false;
                const uint64_t t0 = global_timer_ns();
                for (int spin = 0;; ++spin) {
                    bool mine_ok = true;
                    mk = 0;
                    for (int i = lane; i < a.ncl; i += 32) {
                        const uint64_t *w = gs + size_t(i) * CG_SLOT_WORDS;
                        const uint64_t w0 = ld_relaxed_gpu_u64(w);
                        const uint64_t w1 = ld_relaxed_gpu_u64(w + 1);
                        const uint64_t w2 = ld_relaxed_gpu_u64(w + 2);
                        const uint64_t w3 = ld_relaxed_gpu_u64(w + 3);
                        if ((w0 & 511u) != tag || (w1 & 511u) != tag ||
                            (w2 & 511u) != tag || (w3 & 511u) != tag) {
                            mine_ok = false;
                        } else if (w0 > mk) {
                            mk = w0;
                            mx = __uint_as_float(unsigned(w1 >> 32));
                            my = __uint_as_float(unsigned(w2 >> 32));
                            mz = __uint_as_float(unsigned(w3 >> 32));
                        }
                    }
                    if (__all_sync(FULL, mine_ok)) {
                        ok = true;
                        break;
                    }
                    if ((spin & 63) == 63 && global_timer_ns() - t0 > a.timeout_ns) break;
                }
                if (ok) {
                    // the largest key, and the coordinates that came with it
                    const unsigned mhi = __reduce_max_sync(FULL, unsigned(mk >> 32));
                    const unsigned lo32 = __reduce_max_sync(
                        FULL, unsigned(mk >> 32) == mhi ? unsigned(mk) : 0u);
                    const int wl = __ffs(__ballot_sync(FULL, unsigned(mk >> 32) == mhi &&
                                                                 unsigned(mk) == lo32)) - 1;
                    const float fx = __shfl_sync(FULL, mx, wl);
                    const float fy = __shfl_sync(FULL, my, wl);
                    const float fz = __shfl_sync(FULL, mz, wl);
                    const uint64_t wk = (uint64_t(mhi) << 32) | lo32;
                    const unsigned wj =
                        (FPS_GRID_MAX_N - 1) - unsigned((wk >> 9) & 0xffffffu);
                    // 3. the winner to every block of the cluster
                    if (lane < a.cs) {
                        const uint32_t ra = map_shared_rank(&bslot[par], unsigned(lane));
                        const uint32_t rb = map_shared_rank(&bbar[par], unsigned(lane));
                        st_async_v4(ra, mhi, wj, __float_as_uint(fx), __float_as_uint(fy),
                                    rb);
                        st_async_b32(ra + 16, __float_as_uint(fz), rb);
                    }
                    if (lane == 0 && r == 0) out[t] = int64_t(wj);
                } else if (lane == 0) {
                    raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
                }
            }
        }
        // every block: the winner from the leader
        const bool got = mbar_wait_cluster_bounded(&bbar[par], ph, a.timeout_ns);
        if (threadIdx.x == 0 && got) mbar_arrive_expect_tx(&bbar[par], FPS_CAND_BYTES);
        if (__syncthreads_or(!got)) {
            if (threadIdx.x == 0) raise_status(a.status, 4 /* PC_ERR_DEVICE_TIMEOUT */);
            failed = true;
            break;
        }
        const ClusterSlot w = bslot[par];
        cx = w.x;
        cy = w.y;
        cz = w.z;
    }
    if (failed && r == 0)
        for (int i = t + int(threadIdx.x); i < a.npoint; i += T) out[i] = -1;
    cluster_sync_all();  // no block exits while peers may write
}

// ---------------------------------------------------------------------------
// GRID schedule in rounds (two levels): the rounds above for a cloud spread
// over a cooperative grid of clusters.  Per round:
//   1. every point warp lists its points (as in a cluster) and each block
//      sends its list to its cluster's block 0 (its leader) with one bulk
//      copy into distributed shared memory;
//   2. the leader summarizes its cluster: Bc, the largest bound of its lists;
//      the cluster's largest listed point first; then, in list order, the
//      listed points above Bc, FR_SUM in all (points past that raise Bc to
//      their m, as a block's overflow does); it writes the summary, its
//      length and Bc to the cluster's slot of the workspace and then the
//      round's tag with a release store;
//   3. every block waits for the tags of all clusters of its cloud (acquire;
//      bounded), copies the summaries into shared memory (L2 loads) and
//      certifies the run from them exactly as a cluster certifies it from
//      its blocks' lists: B is the largest Bc, the first center the largest
//      summarized point (the cloud's largest: every warp lists its best and
//      every cluster puts its largest first), later centers the summarized
//      points still strictly above B; every point left out of a summary or
//      of the candidates is at most B.  Positions follow list order, so every
//      block keeps the same candidates and certifies the same run.
// A summary slot is double-buffered by round parity: a leader writes round
// r + 2 only after all its blocks finished round r + 1, which needs every
// cluster's round r + 1 summary, which each cluster publishes only after
// all its blocks finished round r -- so no block still reads round r.
// Every wait is bounded.
constexpr int FR_SUM = 32 * FR_LIST;  // entries of a cluster's summary
constexpr int FR_MAX_LISTS = 64;      // lists or summaries a block scans at most

// A summary slot: FR_SUM entries (32 B), the bound (uint4, key in .x), the
// tag (uint4: round + 1 in .x, the number of entries written in .y).
__host__ __device__ constexpr unsigned fr_sum_bytes() { return FR_SUM * 32u + 32u; }

// Threads of a grid rounds kernel: the point threads and the resolving warp,
// at most 10 warps with 32 points a thread and 12 with 24 (three warps on
// an SM sub-partition leave 168 registers a thread for the points), 13 with
// fewer.
__host__ __device__ constexpr int fgr_max_threads(int ppt) {
    return ppt >= 32 ? 320 : ppt >= 24 ? 384 : 416;
}

// Shared memory: the points, the block's list, the leader's copies of its
// cluster's lists, the cloud's summaries, then the run's state as in
// fps_rounds_smem.
__host__ __device__ constexpr size_t fps_grid_rounds_smem(int chunk, int warps, int cs,
                                                          int ncl) {
    return fr_align16(size_t(chunk) * 12) + fr_msg_bytes(warps) +
           size_t(cs) * fr_msg_bytes(warps) + size_t(ncl) * fr_sum_bytes() +
           size_t(FR_RMAX) * 16 + 32 * FR_LIST * sizeof(int) + 32 * sizeof(uint4) +
           2 * FR_MAX_LISTS * sizeof(int) + 2 * sizeof(uint64_t) + 48;
}

// Workspace of the grid rounds: per cloud [2 parities][ncl] summary slots.
__host__ __device__ constexpr size_t fps_grid_rounds_ws(int64_t B, int ncl) {
    return size_t(B) * 2 * size_t(ncl) * fr_sum_bytes();
}

// When more than CAP - 1 listed entries lie above bnd (*s_total, 1 + their
// number, above CAP = FR_SUM): a bound tau > bnd with at most CAP - 1
// entries above it, as low as two levels of a 64-bin histogram of the keys
// above bnd find; cnt becomes the lists' counts above tau and *s_total 1 +
// their sum.  Dropping the smallest keys keeps a run long, where dropping the
// entries past the first CAP - 1 in list order raises the bound to whatever
// those hold (1M points on 7 clusters: about 50 centers a round instead of
// 13 in a CPU simulation of both rules).  Every thread of the block calls it
// (barriers inside), after fr_count and a barrier; every block computes the
// same bound from the same lists.  hist: 128 ints of shared memory.
__device__ unsigned fr_cap_bound(const unsigned char *lists, int nl, int per, int nscan,
                                 unsigned msg, unsigned bnd, const uint4 *wfirst, int *cnt,
                                 int *hist, int *s_total, unsigned *s_tau, const int *lens) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int CAP = FR_SUM;
    unsigned kmax = lane < nscan ? wfirst[lane].x : 0u;  // the largest key
    kmax = __reduce_max_sync(FULL, kmax);
    const unsigned lo = bnd + 1u;
    const unsigned span = kmax - bnd;  // >= 1: some entry is above bnd
    const int s1 = max(0, 32 - __clz(int(span - 1u)) - 6);  // 64 bins of 2^s1 keys
    const int s2 = max(0, s1 - 6);                           // bin b - 1 in 64 parts
    for (int i = int(threadIdx.x); i < 128; i += int(blockDim.x)) hist[i] = 0;
    __syncthreads();
    auto key_at = [&](int l, int k) {
        return *reinterpret_cast<const unsigned *>(lists + size_t(l) * msg + size_t(k) * 32);
    };
    for (int l = warp; l < nl; l += nscan) {
        const int len = lens ? lens[l] : per;
        for (int k = lane; k < len; k += 32) {
            const unsigned h = key_at(l, k);
            if (h > bnd) atomicAdd(&hist[(h - lo) >> s1], 1);
        }
    }
    __syncthreads();
    // the entries at or above each bin (lane: bins 2 lane, 2 lane + 1), the
    // first bin with at most CAP - 1 of them, and that count
    auto first_fit = [&](const int *hg, int extra, int &b, int &cb) {
        const int h0 = hg[2 * lane], h1 = hg[2 * lane + 1];
        int suf = h0 + h1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_down_sync(FULL, suf, o);
            if (lane + o < 32) suf += v;
        }
        const int c0 = suf + extra, c1 = suf - h0 + extra;
        const unsigned m0 = __ballot_sync(FULL, c0 <= CAP - 1);
        const unsigned m1 = __ballot_sync(FULL, c1 <= CAP - 1);
        b = 64;
        if (m0) b = 2 * (__ffs(m0) - 1);
        if (m1) b = min(b, 2 * (__ffs(m1) - 1) + 1);
        const int v0 = __shfl_sync(FULL, c0, (b >> 1) & 31);
        const int v1 = __shfl_sync(FULL, c1, (b >> 1) & 31);
        cb = b == 64 ? extra : ((b & 1) ? v1 : v0);
    };
    int b, cb;
    first_fit(hist, 0, b, cb);  // b >= 1: bin 0 holds the first too many
    const unsigned base2 = unsigned(b - 1) << s1;
    for (int l = warp; l < nl; l += nscan) {
        const int len = lens ? lens[l] : per;
        for (int k = lane; k < len; k += 32) {
            const unsigned h = key_at(l, k);
            if (h > bnd && ((h - lo) >> s1) == unsigned(b - 1))
                atomicAdd(&hist[64 + (((h - lo) - base2) >> s2)], 1);
        }
    }
    __syncthreads();
    if (warp == 0) {
        int c, cc;
        first_fit(hist + 64, cb, c, cc);
        // every key below lo + base2 + (c << s2) is dropped
        const unsigned long long t =
            (unsigned long long)lo + base2 + ((unsigned long long)c << s2) - 1ull;
        if (lane == 0) *s_tau = unsigned(min(t, (unsigned long long)kmax));
    }
    __syncthreads();
    const unsigned tau = *s_tau;
    for (int l = warp; l < nl; l += nscan) {
        const int len = lens ? lens[l] : per;
        int n = 0;
        for (int k0 = 0; k0 < len; k0 += 32) {
            const int k = k0 + lane;
            n += __popc(__ballot_sync(FULL, k < len && key_at(l, k) > tau));
        }
        if (lane == 0) cnt[l] = n;
    }
    __syncthreads();
    if (warp == 0) {
        const int total = 1 + fr_before(cnt, nl);
        if (lane == 0) *s_total = total;
    }
    __syncthreads();
    return tau;
}

template <int PPT>
__global__ void __launch_bounds__(fgr_max_threads(PPT), 1)
    fps_grid_rounds_kernel(const FpsArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int T = int(blockDim.x) - 32;  // threads holding points
    const int W = T >> 5;                // their warps, which list
    const int NW = W + 1;                // and the resolving warp
    const bool rw = warp == W;
    const unsigned msg = fr_msg_bytes(W);
    const unsigned smsg = fr_sum_bytes();
    float *scoord = reinterpret_cast<float *>(smem);
    unsigned char *sbuf = smem + fr_align16(size_t(a.chunk) * 12);
    unsigned char *recv = sbuf + msg;                          // [cs] lists (leader)
    unsigned char *gsum = recv + size_t(a.cs) * msg;           // [ncl] summaries
    float4 *cen = reinterpret_cast<float4 *>(gsum + size_t(a.ncl) * smsg);
    int *cidx = reinterpret_cast<int *>(cen + FR_RMAX);
    uint4 *wfirst = reinterpret_cast<uint4 *>(cidx + 32 * FR_LIST);
    int *lcnt = reinterpret_cast<int *>(wfirst + 32);  // [FR_MAX_LISTS]
    int *glen = lcnt + FR_MAX_LISTS;  // [FR_MAX_LISTS] entries of each summary
    uint64_t *xbar = reinterpret_cast<uint64_t *>(glen + FR_MAX_LISTS);
    int *s_nc = reinterpret_cast<int *>(xbar + 2);
    int *s_fail = s_nc + 1;
    int *s_total = s_nc + 2;
    unsigned *s_over = reinterpret_cast<unsigned *>(s_nc + 3);
    volatile int *s_pub = s_nc + 4;
    volatile int *s_fin = s_nc + 5;
    int *s_first = s_nc + 6;  // leader: the offset of its cluster's largest entry
    unsigned *s_tau = reinterpret_cast<unsigned *>(s_nc + 7);

    // every distributed-shared-memory address below targets rank 0 of a
    // cluster of a.cs blocks; a launch without that shape stops here
    if (cluster_nctarank() != unsigned(a.cs) || a.cs > FR_MAX_LISTS ||
        a.ncl > FR_MAX_LISTS) {
        if (threadIdx.x == 0) raise_status(a.status, 3 /* PC_ERR_CUDA */);
        return;
    }
    const unsigned rank = cluster_ctarank();
    const int b = blockIdx.x / a.nblocks;
    const int r = blockIdx.x % a.nblocks;  // block of the cloud
    const int cl = r / a.cs;               // cluster of the cloud
    const float *x = a.xyz + size_t(b) * size_t(a.N) * 3;
    const int lo = r * a.chunk;
    const int hi = min(a.N, lo + a.chunk);
    const float2 nz0 = make_float2(a.negzero, a.negzero);
    const unsigned xbytes = unsigned(a.cs) * msg;
    // slot (parity p, cluster c) of this cloud
    unsigned char *ws = reinterpret_cast<unsigned char *>(a.slots) +
                        size_t(b) * 2 * size_t(a.ncl) * smsg;
    auto slot = [&](int p, int c) { return ws + (size_t(p) * a.ncl + c) * smsg; };

    ThreadPoints<PPT> pt;
    if (!rw) {
        fps_load_points<PPT>(x, lo, hi, T, pt, scoord);
    } else {
#pragma unroll
        for (int p = 0; p < PPT; ++p) pt.m[p] = -1.0f;
#pragma unroll
        for (int i = 0; i < PPT / 2; ++i) pt.x[i] = pt.y[i] = pt.z[i] = make_float2(0.f, 0.f);
    }
    int64_t *out = a.out + size_t(b) * a.npoint;
    if (threadIdx.x == 0) {
        cen[0] = make_float4(x[size_t(a.start) * 3 + 0], x[size_t(a.start) * 3 + 1],
                             x[size_t(a.start) * 3 + 2], 0.f);
        *s_nc = 1;
        *s_fail = 0;
        *s_total = 1;
        *s_over = 0u;
        *s_pub = 0;
        *s_fin = 0;
        if (r == 0) out[0] = a.start;
        // the leader's exchange mbarriers, one per round parity
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (rank == 0) {
            mbar_arrive_expect_tx(&xbar[0], xbytes);
            mbar_arrive_expect_tx(&xbar[1], xbytes);
        }
    }
    __syncthreads();
    cluster_sync_all();  // the leader's barriers exist before any copy

    auto apply = [&](const float4 cc) {
        const float2 ncx = make_float2(-cc.x, -cc.x);
        const float2 ncy = make_float2(-cc.y, -cc.y);
        const float2 ncz = make_float2(-cc.z, -cc.z);
#pragma unroll
        for (int i = 0; i < PPT / 2; ++i) {
            const float2 s = sqdist2(pt.x[i], pt.y[i], pt.z[i], ncx, ncy, ncz, nz0);
            pt.m[2 * i] = fminf(pt.m[2 * i], s.x);
            pt.m[2 * i + 1] = fminf(pt.m[2 * i + 1], s.y);
        }
    };
    // lower them by two centers at once (min is exact in any order)
    auto apply2 = [&](const float4 c0, const float4 c1) {
        const float2 ncx = make_float2(-c0.x, -c0.x);
        const float2 ncy = make_float2(-c0.y, -c0.y);
        const float2 ncz = make_float2(-c0.z, -c0.z);
        const float2 mcx = make_float2(-c1.x, -c1.x);
        const float2 mcy = make_float2(-c1.y, -c1.y);
        const float2 mcz = make_float2(-c1.z, -c1.z);
#pragma unroll
        for (int i = 0; i < PPT / 2; ++i) {
            const float2 s = sqdist2(pt.x[i], pt.y[i], pt.z[i], ncx, ncy, ncz, nz0);
            const float2 u = sqdist2(pt.x[i], pt.y[i], pt.z[i], mcx, mcy, mcz, nz0);
            pt.m[2 * i] = fmin3(pt.m[2 * i], s.x, u.x);
            pt.m[2 * i + 1] = fmin3(pt.m[2 * i + 1], s.y, u.y);
        }
    };
    FrEntry *mine = reinterpret_cast<FrEntry *>(sbuf) + warp * FR_CW;
    uint4 *mybound = reinterpret_cast<uint4 *>(sbuf + size_t(W) * FR_CW * 32) + warp;
    int t = 1;  // centers output so far
    for (int round = 0; t < a.npoint; ++round) {
        const int par = round & 1;
        const unsigned tag = unsigned(round) + 1u;
        if (round == 0 && !rw) apply(cen[0]);
        if (!rw) fr_list<PPT>(pt, scoord, lo, T, mine, mybound);
        fence_proxy_async_smem();  // the list, for the bulk copy
        __syncthreads();
        // 1. the block's list to its leader; the list may be rewritten once
        // the copy has read it
        if (rw && lane == 0) {
            const uint32_t dst = map_shared_rank(recv + size_t(rank) * msg, 0u);
            const uint32_t bar = map_shared_rank(&xbar[par], 0u);
            bulk_copy_to_cluster(dst, sbuf, msg, bar);
            bulk_commit();
            bulk_wait_read_all();
        }
        // 2. the leader: its cluster's summary, then the round's tag
        if (rank == 0) {
            const unsigned ph = unsigned(round >> 1) & 1u;
            const bool got =
                __all_sync(FULL, mbar_wait_cluster_bounded(&xbar[par], ph, a.timeout_ns));
            if (threadIdx.x == 0 && got) mbar_arrive_expect_tx(&xbar[par], xbytes);
            if (!got && lane == 0) *s_fail = 1;
            __syncthreads();
            if (!*s_fail) {
                unsigned bc =
                    fr_count(recv, a.cs, W * FR_CW, W, NW, msg, lcnt, wfirst + warp);
                __syncthreads();
                if (warp == 0) {  // the cluster's largest entry and the candidates' count
                    const uint4 f = lane < NW ? wfirst[lane] : make_uint4(0u, FULL, 0u, 0u);
                    unsigned fh, fj;
                    warp_argmax_hi_min_lo(f.x, f.y, fh, fj);
                    const int who = __ffs(__ballot_sync(FULL, f.x == fh && f.y == fj)) - 1;
                    const int off = int(__shfl_sync(FULL, f.z, who));
                    const int total = 1 + fr_before(lcnt, a.cs);
                    if (lane == 0) {
                        *s_first = fh != 0u ? off : -1;
                        *s_total = total;
                    }
                }
                __syncthreads();
                // more candidates than a summary holds: drop the smallest
                if (*s_total > FR_SUM)
                    bc = fr_cap_bound(recv, a.cs, W * FR_CW, NW, msg, bc, wfirst, lcnt, cidx,
                                      s_total, s_tau, nullptr);
                fr_place(recv, a.cs, W * FR_CW, NW, msg, bc, lcnt, cidx, s_over);
                __syncthreads();
                unsigned char *sl = slot(par, cl);
                const int first = *s_first;
                const int total = *s_total;
                const int n = min(total, FR_SUM);  // positions written
                for (int e = int(threadIdx.x); e < n; e += int(blockDim.x)) {
                    int off = e == 0 ? first : (e < total ? cidx[e] : -1);
                    if (e > 0 && off == first) off = -1;  // already at position 0
                    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
                    if (off >= 0) {
                        v0 = reinterpret_cast<const uint4 *>(recv + off)[0];
                        v1 = reinterpret_cast<const uint4 *>(recv + off)[1];
                    }
                    reinterpret_cast<uint4 *>(sl + size_t(e) * 32)[0] = v0;
                    reinterpret_cast<uint4 *>(sl + size_t(e) * 32)[1] = v1;
                }
                if (threadIdx.x == 0) {
                    *reinterpret_cast<uint4 *>(sl + FR_SUM * 32) =
                        make_uint4(max(bc, *s_over), 0u, 0u, 0u);
                    reinterpret_cast<unsigned *>(sl + FR_SUM * 32 + 16)[1] = unsigned(n);
                }
                __syncthreads();
                // testing hook: cluster 0 of the first cloud withholds round 0
                const bool withhold = (a.stall & 1) && b == 0 && cl == 0 && round == 0;
                // the block's writes, ordered by the barrier, are released with
                // the tag
                if (threadIdx.x == 0 && !withhold)
                    st_release_gpu_u32(reinterpret_cast<unsigned *>(sl + FR_SUM * 32 + 16),
                                       tag);
            }
        }
        // 3. every block: the round's summaries of all clusters of the cloud
        if (rw && !*s_fail) {
            bool ok = true;
            for (int c = lane; c < a.ncl && ok; c += 32) {
                const unsigned *tp =
                    reinterpret_cast<const unsigned *>(slot(par, c) + FR_SUM * 32 + 16);
                const uint64_t t0 = global_timer_ns();
                for (int spin = 0;; ++spin) {
                    if (ld_acquire_gpu_u32(tp) == tag) break;
                    if ((spin & 63) == 63 && global_timer_ns() - t0 > a.timeout_ns) {
                        ok = false;
                        break;
                    }
                }
                if (ok) glen[c] = min(int(__ldcg(tp + 1)), FR_SUM);
            }
            if (!__all_sync(FULL, ok) && lane == 0) *s_fail = 1;
        }
        __syncthreads();
        if (!*s_fail) {  // each summary's entries and bound (a warp per summary)
            for (int c = warp; c < a.ncl; c += NW) {
                const uint4 *src = reinterpret_cast<const uint4 *>(slot(par, c));
                uint4 *dst = reinterpret_cast<uint4 *>(gsum + size_t(c) * smsg);
                const int n16 = 2 * glen[c];
                for (int v = lane; v < n16; v += 32) dst[v] = __ldcg(src + v);
                if (lane == 0) dst[2 * FR_SUM] = __ldcg(src + 2 * FR_SUM);
            }
        }
        if (threadIdx.x == 0) {  // the leader's counters, for the cloud's candidates
            *s_total = 1;
            *s_over = 0u;
        }
        __syncthreads();
        if (!*s_fail) {
            // 4. the cloud's candidates and the run, as in fps_rounds_kernel
            unsigned bnd =
                fr_count(gsum, a.ncl, FR_SUM, 1, NW, smsg, lcnt, wfirst + warp, glen);
            __syncthreads();
            if (warp == 0) {
                const int total = 1 + fr_before(lcnt, a.ncl);
                if (lane == 0) *s_total = total;
            }
            __syncthreads();
            // more candidates than the resolving warp holds: drop the smallest
            if (*s_total > FR_SUM)
                bnd = fr_cap_bound(gsum, a.ncl, FR_SUM, NW, smsg, bnd, wfirst, lcnt, cidx,
                                   s_total, s_tau, glen);
            fr_place(gsum, a.ncl, FR_SUM, NW, smsg, bnd, lcnt, cidx, s_over, glen);
            __syncthreads();
            if (rw) {
                fr_pick(gsum, NW, bnd, min(FR_RMAX, a.npoint - t), cidx, wfirst, *s_total,
                        *s_over, cen, s_nc, s_pub, s_fin, r == 0 ? out + t : nullptr);
            } else {
                // (a warp that finds nothing new sleeps briefly instead of polling:
                // its loads and fences would slow the resolving warp's shuffles)
                int c = 0;
                const uint64_t w0 = global_timer_ns();
                for (int spin = 0;; ++spin) {
                    const int fin = *s_fin;
                    const int pub = *s_pub;
                    if (pub > c || fin) {
                        __threadfence_block();  // the centers published before pub / fin
                        const int upto = fin ? *s_pub : pub;
                        while (c < upto) {  // two at a time where two are out
                            if (c + 1 < upto) {
                                apply2(cen[c], cen[c + 1]);
                                c += 2;
                            } else {
                                apply(cen[c]);
                                ++c;
                            }
                        }
                        if (fin) break;
                        continue;
                    }
                    __nanosleep(32);
                    if ((spin & 63) == 63 && global_timer_ns() - w0 > a.timeout_ns) {
                        if (lane == 0) *s_fail = 1;
                        break;
                    }
                }
            }
            __syncthreads();
        }
        const int taken = *s_nc;
        if (*s_fail || taken <= 0) {
            raise_status(a.status, *s_fail ? 4 /* PC_ERR_DEVICE_TIMEOUT */ : 3 /* PC_ERR_CUDA */);
            if (r == 0)
                for (int i = t + int(threadIdx.x); i < a.npoint; i += int(blockDim.x)) out[i] = -1;
            break;
        }
        t += taken;
        if (threadIdx.x == 0) {  // for the next round
            *s_total = 1;
            *s_over = 0u;
            *s_pub = 0;
            *s_fin = 0;
        }
    }
    // no copy in flight and no block exits while peers may write
    if (rw && lane == 0) bulk_wait_all();
    cluster_sync_all();
}

template <int PPT>
const void *fgr_ptr_t() {
    return reinterpret_cast<const void *>(&fps_grid_rounds_kernel<PPT>);
}

const void *fps_grid_rounds_ptr(int ppt) {
    switch (ppt) {
        case 2: return fgr_ptr_t<2>();
        case 4: return fgr_ptr_t<4>();
        case 8: return fgr_ptr_t<8>();
        case 16: return fgr_ptr_t<16>();
        case 24: return fgr_ptr_t<24>();
        default: return fgr_ptr_t<32>();
    }
}

const void *fps_rounds_ptr(int ppt) {
    switch (ppt) {
        case 2: return reinterpret_cast<const void *>(&fps_rounds_kernel<2>);
        case 4: return reinterpret_cast<const void *>(&fps_rounds_kernel<4>);
        case 8: return reinterpret_cast<const void *>(&fps_rounds_kernel<8>);
        case 16: return reinterpret_cast<const void *>(&fps_rounds_kernel<16>);
        case 24: return reinterpret_cast<const void *>(&fps_rounds_kernel<24>);
        default: return reinterpret_cast<const void *>(&fps_rounds_kernel<32>);
    }
}

template <int PPT>
const void *cluster_kernel_ptr(bool cluster) {
    return cluster ? reinterpret_cast<const void *>(&fps_cluster_kernel<PPT, true>)
                   : reinterpret_cast<const void *>(&fps_cluster_kernel<PPT, false>);
}

constexpr int kPptChoices[] = {2, 4, 8, 16, 24, 32};

const void *fps_kernel_ptr(int strategy, int ppt) {
    const bool cl = strategy == 2;
    if (strategy == 3) {
        switch (ppt) {
            case 2: return reinterpret_cast<const void *>(&fps_grid_kernel<2>);
            case 4: return reinterpret_cast<const void *>(&fps_grid_kernel<4>);
            case 8: return reinterpret_cast<const void *>(&fps_grid_kernel<8>);
            case 16: return reinterpret_cast<const void *>(&fps_grid_kernel<16>);
            case 24: return reinterpret_cast<const void *>(&fps_grid_kernel<24>);
            default: return reinterpret_cast<const void *>(&fps_grid_kernel<32>);
        }
    }
    switch (ppt) {
        case 2: return cluster_kernel_ptr<2>(cl);
        case 4: return cluster_kernel_ptr<4>(cl);
        case 8: return cluster_kernel_ptr<8>(cl);
        case 16: return cluster_kernel_ptr<16>(cl);
        case 24: return cluster_kernel_ptr<24>(cl);
        default: return cluster_kernel_ptr<32>(cl);
    }
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

// Points per thread and threads for a block holding `chunk` points: the
// fewest points per thread that keep the block at or below `target` threads
// (about eight warps keep the per-step reductions short); if no choice gets
// there, the most threads the largest choice allows.  Returns false when the
// chunk does not fit at all.
bool pick_shape(int chunk, int target, int &ppt, int &threads) {
    for (int p : kPptChoices) {
        const int t = std::max(32, round_up((chunk + p - 1) / p, 32));
        if (t <= target && t <= fps_max_threads(p)) {
            ppt = p;
            threads = t;
            return true;
        }
    }
    for (int p : kPptChoices) {
        const int t = std::max(32, round_up((chunk + p - 1) / p, 32));
        if (t <= fps_max_threads(p)) {
            ppt = p;
            threads = t;
            return true;
        }
    }
    return false;
}

int64_t block_capacity() {
    int64_t c = 0;
    for (int p : kPptChoices) c = std::max<int64_t>(c, int64_t(p) * fps_max_threads(p));
    return c;
}

// Threads per block the planner aims for: measured on GB300 (100k-point
// cloud on a 16-block cluster: 0.84 us per step at 256 threads, 0.88 at 512,
// 0.99 at 128 and at 1024).
constexpr int kTargetThreads = 256;

// Clusters of `cs` blocks of kernel `fn` (threads, dynamic shared memory)
// that can be resident at once: cudaOccupancyMaxActiveClusters, 0 when none
// or when the query fails.
int max_active_clusters(const void *fn, int cs, int threads, size_t smem) {
    if (cs > 8 &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(smem)) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(cs));
    cfg.blockDim = dim3(unsigned(threads));
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

bool cluster_fits(const DeviceInfo &dev, int cs, int threads, size_t smem,
                  int ppt) {
    (void)dev;
    return max_active_clusters(fps_kernel_ptr(2, ppt), cs, threads, smem) >= 1;
}

size_t cluster_smem(int chunk) {
    return fps_coords_bytes(chunk) + 32 * sizeof(uint2) +
           2 * FPS_MAX_CLUSTER * sizeof(ClusterSlot) + 2 * sizeof(uint64_t) + 16;
}

// The two-level grid kernel adds the winner's mbarrier pair and slots.
size_t cgrid_smem(int chunk) {
    return cluster_smem(chunk) + 2 * sizeof(uint64_t) + 2 * sizeof(ClusterSlot);
}

const void *fps_cgrid_ptr(int ppt) {
    switch (ppt) {
        case 2: return reinterpret_cast<const void *>(&fps_cgrid_kernel<2>);
        case 4: return reinterpret_cast<const void *>(&fps_cgrid_kernel<4>);
        case 8: return reinterpret_cast<const void *>(&fps_cgrid_kernel<8>);
        case 16: return reinterpret_cast<const void *>(&fps_cgrid_kernel<16>);
        case 24: return reinterpret_cast<const void *>(&fps_cgrid_kernel<24>);
        default: return reinterpret_cast<const void *>(&fps_cgrid_kernel<32>);
    }
}

// The two-level GRID plan for clusters of `cs` blocks: with bpc_req > 0 that
// many blocks per cloud (a multiple of cs), else as many clusters as can be
// resident with every cloud holding the same number.  p.ok = false when the
// clusters cannot all be resident.
FpsPlan plan_cgrid(const DeviceInfo &dev, int64_t B, int64_t N, int cs, int bpc_req) {
    FpsPlan p;
    p.strategy = 3;
    p.cluster = cs;
    if (bpc_req > 0 && bpc_req % cs != 0) {
        p.why = "blocks_per_cloud is not a multiple of the cluster size";
        return p;
    }
    const int nsm = std::max(1, dev.sm_count);
    int64_t bpc = bpc_req > 0 ? bpc_req : (nsm / std::max<int64_t>(B, 1)) / cs * cs;
    for (int iter = 0; iter < 3 && bpc >= cs; ++iter) {
        if (bpc > N) bpc = std::max<int64_t>(cs, N / cs * cs);
        p.chunk = int((N + bpc - 1) / bpc);
        if (!pick_shape(p.chunk, kTargetThreads, p.ppt, p.threads)) {
            p.why = "cloud too large for the on-chip FPS schedules";
            return p;
        }
        p.smem_bytes = cgrid_smem(p.chunk);
        if (p.smem_bytes > dev.smem_per_block_optin) {
            p.why = "block's share of the cloud exceeds shared memory";
            return p;
        }
        const int n = max_active_clusters(fps_cgrid_ptr(p.ppt), cs, p.threads,
                                          p.smem_bytes);
        const int64_t ncl_fit = n / std::max<int64_t>(B, 1);
        if (ncl_fit * cs >= bpc) {
            if (bpc_req > 0 || ncl_fit * cs == bpc) {
                p.blocks_per_cloud = int(bpc);
                // 8 words per cluster and cloud; sized as the one-level
                // schedule's 2 words per block when that is more (cs >= 4),
                // so that the size does not depend on the cluster chosen
                const size_t words =
                    size_t(B) * std::max<size_t>(2 * CG_SLOT_WORDS * size_t(bpc / cs),
                                                 2 * size_t(bpc));
                p.workspace_bytes = (words * sizeof(uint64_t) + 255) & ~size_t(255);
                p.step_workspace_bytes = p.workspace_bytes;
                // in rounds: the same blocks with a resolving warp more, where
                // its shared memory fits and every cluster stays resident
                // (the step's shape, else 32 points a thread where the
                // resolving warp would leave too few registers)
                const int ncl = int(bpc / cs);
                int rppt = p.ppt, rthreads = p.threads + 32;
                if (rthreads > fgr_max_threads(rppt)) {
                    rppt = 32;
                    rthreads = std::max(32, round_up((p.chunk + 31) / 32, 32)) + 32;
                }
                const size_t rsmem =
                    fps_grid_rounds_smem(p.chunk, rthreads / 32 - 1, cs, ncl);
                if (rthreads <= fgr_max_threads(rppt) && ncl <= FR_MAX_LISTS &&
                    cs <= FR_MAX_LISTS && rsmem <= dev.smem_per_block_optin &&
                    max_active_clusters(fps_grid_rounds_ptr(rppt), cs, rthreads, rsmem) /
                            std::max<int64_t>(B, 1) >= ncl) {
                    p.grid_rounds = true;
                    p.rounds_ppt = rppt;
                    p.rounds_threads = rthreads;
                    p.rounds_smem = rsmem;
                    p.workspace_bytes = std::max(
                        p.workspace_bytes, (fps_grid_rounds_ws(B, ncl) + 255) & ~size_t(255));
                }
                p.ok = true;
                return p;
            }
        }
        if (bpc_req > 0 || ncl_fit == 0) break;
        bpc = ncl_fit * cs;  // as many as fit with this shape; check again
    }
    p.why = "two-level grid clusters cannot all be resident";
    return p;
}

FpsPlan plan_fps_uncached(const DeviceInfo &dev, int64_t B, int64_t N, int strategy,
                          int cluster_size, int blocks_per_cloud);

}  // namespace

// Plans depend only on the device and the arguments; the occupancy queries
// behind them cost host time on every call, so they are kept (each process
// sees few distinct shapes).
FpsPlan plan_fps(const DeviceInfo &dev, int64_t B, int64_t N, int strategy,
                 int cluster_size, int blocks_per_cloud) {
    using Key = std::tuple<int, int64_t, int64_t, int, int, int>;
    static std::mutex mu;
    static std::map<Key, FpsPlan> cache;
    const Key key{dev.device, B, N, strategy, cluster_size, blocks_per_cloud};
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const FpsPlan p = plan_fps_uncached(dev, B, N, strategy, cluster_size, blocks_per_cloud);
    std::lock_guard<std::mutex> lock(mu);
    if (cache.size() < 4096) cache.emplace(key, p);
    return p;
}

namespace {

FpsPlan plan_fps_uncached(const DeviceInfo &dev, int64_t B, int64_t N, int strategy,
                          int cluster_size, int blocks_per_cloud) {
    FpsPlan p;
    const int64_t cap_block = block_capacity();
    const int nsm = std::max(1, dev.sm_count);
    if (strategy == 0) {  // automatic
        if (N <= 2048 || (B >= nsm / 2 && N <= cap_block))
            strategy = 1;
        else if (N <= cap_block * FPS_MAX_CLUSTER)
            strategy = 2;
        else
            strategy = 3;
    }
    p.strategy = strategy;
    if (strategy == 1 || strategy == 2) {
        int cs = 1;
        if (strategy == 2) {
            if (cluster_size > 0) {
                cs = cluster_size;
            } else {
                cs = 1;
                while (cs < FPS_MAX_CLUSTER && int64_t(cs) * cap_block < N) cs *= 2;
                while (cs < FPS_MAX_CLUSTER && B * (cs * 2) <= nsm &&
                       N / (cs * 2) >= 1024)
                    cs *= 2;
            }
            if (cs < 1 || cs > FPS_MAX_CLUSTER) {
                p.why = "cluster size must be 1..16";
                return p;
            }
        }
        p.cluster = cs;
        p.blocks_per_cloud = cs;
        p.chunk = int((N + cs - 1) / cs);
        if (!pick_shape(p.chunk, kTargetThreads, p.ppt, p.threads)) {
            p.why = "cloud too large for one block/cluster schedule";
            return p;
        }
        p.smem_bytes = cluster_smem(p.chunk);
        if (p.smem_bytes > dev.smem_per_block_optin) {
            p.why = "block's share of the cloud exceeds shared memory";
            return p;
        }
        // When the schedule fits in one wave, each block claims its SM's whole
        // shared memory: blocks of kernels running concurrently on other
        // streams then cannot share an FPS SM and slow its per-step latency.
        if (B * cs <= nsm)
            p.smem_bytes = std::max(p.smem_bytes, dev.smem_per_block_optin);
        if (strategy == 2 && !cluster_fits(dev, cs, p.threads, p.smem_bytes, p.ppt)) {
            if (cluster_size > 0 || cs <= 8) {
                p.why = "cluster of this size cannot be resident on this device";
                return p;
            }
            // 16-block clusters unavailable: retry with 8 or the grid schedule
            if (N <= cap_block * 8)
                return plan_fps(dev, B, N, 2, 8, 0);
            return plan_fps(dev, B, N, 3, 0, 0);
        }
        p.ok = true;
        return p;
    }
    if (strategy == 3) {
        if (N >= FPS_GRID_MAX_N) {
            p.why = "grid schedule supports N < 2^24";
            return p;
        }
        if (!dev.cooperative) {
            p.why = "device has no cooperative launch";
            return p;
        }
        // two levels (clusters exchanging through distributed shared memory,
        // then one slot per cluster in the workspace) unless cluster_size is
        // 1: the cluster size that keeps the most blocks resident
        if (cluster_size != 1) {
            // one center per exchange: the largest cluster that fits, fewest
            // slots and leaders in the global exchange (GB300, 1M points: 2.0
            // us per step with 7 clusters of 16, 2.7 with 15 of 8, 6.9 with
            // 36 of 4, when every block polled every slot).  In rounds the
            // exchange is paid once a run and the point work per center
            // counts more: the size whose rounds plan holds the most blocks
            // (1M points, 16,384 samples: 9.3 ms on 15 clusters of 8, 10.5
            // on 7 of 16)
            FpsPlan best, first;
            const int sizes[3] = {16, 8, 4};
            for (int cs : sizes) {
                if (cluster_size > 1 && cs != cluster_size) continue;
                const FpsPlan c = plan_cgrid(dev, B, N, cs, blocks_per_cloud);
                if (!c.ok) continue;
                if (!first.ok) first = c;
                if (c.grid_rounds &&
                    (!best.ok || c.blocks_per_cloud > best.blocks_per_cloud))
                    best = c;
            }
            if (!best.ok) best = first;
            if (cluster_size > 1 && !best.ok && cluster_size != 16 &&
                cluster_size != 8 && cluster_size != 4)
                best = plan_cgrid(dev, B, N, cluster_size, blocks_per_cloud);
            if (best.ok) return best;
            if (cluster_size > 1) {
                p.why = "two-level grid with this cluster size cannot be resident";
                return p;
            }
        }
        int bpc = blocks_per_cloud;
        if (bpc <= 0) bpc = int(std::max<int64_t>(1, nsm / std::max<int64_t>(B, 1)));
        bpc = int(std::min<int64_t>(bpc, N));
        if (int64_t(bpc) * B > nsm) {
            p.why = "grid schedule needs blocks_per_cloud * B <= SM count";
            return p;
        }
        p.blocks_per_cloud = bpc;
        p.cluster = 1;
        p.chunk = int((N + bpc - 1) / bpc);
        if (!pick_shape(p.chunk, kTargetThreads, p.ppt, p.threads)) {
            p.why = "cloud too large for the on-chip FPS schedules";
            return p;
        }
        p.smem_bytes = 0;
        p.workspace_bytes = (size_t(B) * 2 * bpc * sizeof(uint64_t) + 255) & ~size_t(255);
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, fps_kernel_ptr(3, p.ppt), p.threads, 0) != cudaSuccess) {
            cudaGetLastError();
            p.why = "occupancy query failed";
            return p;
        }
        if (int64_t(per_sm) * nsm < int64_t(bpc) * B) {
            p.why = "grid schedule blocks cannot all be resident";
            return p;
        }
        p.ok = true;
        return p;
    }
    p.why = "unknown FPS strategy";
    return p;
}

}  // namespace

cudaError_t launch_fps(const DeviceInfo &dev, const FpsPlan &plan,
                       const float *xyz, int64_t B, int64_t N, int64_t npoint,
                       int64_t start_idx, int64_t *out_idx, void *workspace,
                       cudaStream_t stream) {
    FpsArgs a{};
    a.xyz = xyz;
    a.N = int(N);
    a.npoint = int(npoint);
    a.start = int(start_idx);
    a.out = out_idx;
    a.chunk = plan.chunk;
    a.nblocks = plan.blocks_per_cloud;
    a.cs = plan.strategy == 3 ? plan.cluster : 1;
    a.ncl = plan.blocks_per_cloud / std::max(1, a.cs);
    a.slots = static_cast<uint64_t *>(workspace);
    a.status = dev.status_word;
    a.timeout_ns = wait_timeout_ns();
    a.stall = debug_stall();
    a.negzero = -0.0f;

    const bool cgrid = plan.strategy == 3 && plan.cluster > 1;
    // two-level GRID in rounds (fps_grid_rounds_kernel) where the plan allows
    const bool grounds = cgrid && plan.grid_rounds && fps_batched();
    const void *fn = grounds  ? fps_grid_rounds_ptr(plan.rounds_ppt)
                     : cgrid ? fps_cgrid_ptr(plan.ppt)
                             : fps_kernel_ptr(plan.strategy, plan.ppt);
    size_t smem = grounds ? plan.rounds_smem : plan.smem_bytes;
    // CLUSTER: several centers per exchange (fps_rounds_kernel) where its
    // lists fit; the step-by-step kernel otherwise.  (With one block per
    // cloud there is no exchange to share: one center per step is faster --
    // GB300, 96 clouds of 4096 points, 1024 samples: 0.41 ms vs 0.54.)
    unsigned threads = unsigned(grounds ? plan.rounds_threads : plan.threads);
    if (fps_batched() && plan.strategy == 2 && plan.threads + 32 <= fr_max_threads(plan.ppt)) {
        const size_t need = fps_rounds_smem(plan.chunk, plan.threads / 32, plan.cluster);
        const size_t rsmem = std::max(smem, need);
        const void *rfn = fps_rounds_ptr(plan.ppt);
        if (rsmem <= dev.smem_per_block_optin &&
            max_active_clusters(rfn, plan.cluster, plan.threads + 32, rsmem) >= 1) {
            fn = rfn;
            smem = rsmem;
            threads = unsigned(plan.threads + 32);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(B * plan.blocks_per_cloud));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    void *args[] = {&a};
    cudaError_t e;
    if (cgrid) {
        e = cudaMemsetAsync(workspace, 0, plan.workspace_bytes, stream);
        if (e != cudaSuccess) return e;
        if (plan.cluster > 8) {
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(plan.cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        // cooperative: every cluster resident at once, or no launch; where
        // the runtime refuses cooperative cluster launches, the plan's
        // occupancy check alone stands behind co-residency (and every wait
        // is bounded)
        attr[1].id = cudaLaunchAttributeCooperative;
        attr[1].val.cooperative = 1;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelExC(&cfg, fn, args);
        if (e != cudaSuccess) {
            cudaGetLastError();
            cfg.numAttrs = 1;
            e = cudaLaunchKernelExC(&cfg, fn, args);
        }
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (plan.strategy == 3) {
        e = cudaMemsetAsync(workspace, 0, plan.workspace_bytes, stream);
        if (e != cudaSuccess) return e;
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.numAttrs = 1;
    } else {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        if (plan.strategy == 2) {
            if (plan.cluster > 8) {
                e = cudaFuncSetAttribute(
                    fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
                if (e != cudaSuccess) return e;
            }
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = unsigned(plan.cluster);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.numAttrs = 1;
        }
    }
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace pcn
