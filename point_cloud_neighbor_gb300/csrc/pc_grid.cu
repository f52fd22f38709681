// pc_grid.cu -- exact grid-accelerated kNN and Ball Query on sm_103a.
//
// The mps-pointops project page's "Roadmap" (Phase 4) calls for spatial
// acceleration structures (a uniform grid or BVH) for large clouds.  This
// file builds a uniform grid over each reference cloud on the GPU and
// answers kNN and Ball Query queries from it with exactly the results of the
// brute-force operators (pc_knn.cu, pc_ball_query.cu): the same separately
// rounded squared distance, the same (s, j) order and strict radius test.
//
// Build (pc_grid_build), per cloud:
//   1. bounds: order-preserving integer keys of min/max per axis (warp
//      reductions + atomics);
//   2. D cells per axis (D^3 ~ N / 4, fixed from N on the host), cell size
//      h = extent / D; cell of a point: floor(fl(fl(x - lo) * inv_h)),
//      clamped to [0, D-1];
//   3. per-cell counts, exclusive scan, scatter: the points in cell order as
//      float4 (x, y, z, original index), so every x-row of cells is one
//      contiguous range.
// Query (one warp per query): kNN searches cubes of cells of growing
// half-width R around the query's cell, a shell at a time, and stops once the
// cube holds every cell that can contain a point with s <= tau (tau: the
// current k-th squared distance).  Ball Query examines the cells that can
// hold a point with s < fl(r^2) and keeps the K smallest indices among the
// hits.  Candidates are inserted into warp-distributed sorted lists (lane l
// holds entries l, l + 32, ...).
//
// Exactness: the cell of a coordinate, floor(fl(fl(x - lo) * inv_h)) clamped,
// is monotone in x.  A point with s32 <= rho^2 has |x - q| <= rho (1 + 3u) +
// 6.5e-23 on every axis (u = 2^-24; the absolute term covers squares that
// round below the normal range), so it lies between the cells of the floats
// q - reach and q + reach once reach exceeds that bound by the rounding of
// q -+ reach: reach = rho (1 + 1e-5) + 1e-5 (|qx| + |qy| + |qz|) + 1e-22.
// The same cell function and header serve the build and the queries, so no
// face of a cell is ever computed.
#include "pointcloud.h"
#include "pc_device.cuh"
#include "pc_internal.h"

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>

namespace pcn {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kTargetPerCell = 4;
constexpr int kMaxD = 256;
constexpr int kMaxKGrid = 256;

struct __align__(16) GridHeader {  // 128 bytes per cloud
    unsigned kmin[3], kmax[3];     // order-preserving keys of the bounds
    float lo[3];
    float inv_h[3];
    int D;
    int pad[17];
};
static_assert(sizeof(GridHeader) == 128, "grid header size");

struct GridGeometry {
    int D = 1;
    int64_t C = 1;
    size_t off_header = 0, off_start = 0, off_count = 0, off_pts = 0, total = 0;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

GridGeometry grid_geometry(int64_t B, int64_t N) {
    GridGeometry g;
    int D = int(std::lround(std::cbrt(double(std::max<int64_t>(N, 1)) / kTargetPerCell)));
    g.D = std::min(kMaxD, std::max(1, D));
    g.C = int64_t(g.D) * g.D * g.D;
    g.off_header = 0;
    g.off_start = align256(size_t(B) * sizeof(GridHeader));
    g.off_count = g.off_start + align256(size_t(B) * size_t(g.C + 1) * 4);
    g.off_pts = g.off_count + align256(size_t(B) * size_t(g.C) * 4);
    g.total = g.off_pts + align256(size_t(B) * size_t(N) * 16);
    return g;
}

struct GridView {
    const GridHeader *hdr;
    const int *start;     // [B][C + 1]
    const float4 *pts;    // [B][N]
    int D;
    int64_t C;
    int N;
};

GridView grid_view(const void *grid, int64_t B, int64_t N) {
    const GridGeometry g = grid_geometry(B, N);
    const unsigned char *base = static_cast<const unsigned char *>(grid);
    GridView v;
    v.hdr = reinterpret_cast<const GridHeader *>(base + g.off_header);
    v.start = reinterpret_cast<const int *>(base + g.off_start);
    v.pts = reinterpret_cast<const float4 *>(base + g.off_pts);
    v.D = g.D;
    v.C = g.C;
    v.N = int(N);
    return v;
}

__device__ __forceinline__ unsigned order_key(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ int cell_axis(float x, float lo, float inv_h, int D) {
    const float t = __fmul_rn(__fsub_rn(x, lo), inv_h);
    return min(max(__float2int_rd(t), 0), D - 1);
}

// Slack added to a real radius r before it is turned into a range of cells
// around a query q: 1e-5 r + 1e-5 (|qx| + |qy| + |qz|) + 1e-22.  It covers
// (a) s32 >= s (1 - 5u) - 5 * 2^-150 (three roundings of squares and two of
// sums, absolute error below the normal range), i.e. |dx| <= sqrt(s32)
// (1 + 3u) + 6.5e-23 for every point with s32 <= r^2, and (b) the rounding of
// q -+ reach and of the slack itself (u = 2^-24 each).
__device__ __forceinline__ float query_slack(float qx, float qy, float qz) {
    return 1e-5f * (fabsf(qx) + fabsf(qy) + fabsf(qz)) + 1e-22f;
}

// Cells [c0, c1] along one axis that hold every reference point x with
// |x - q| <= reach_needed: cell_axis is monotone in x, so the cells of the
// floats q - reach and q + reach (each rounded outwards of the needed range
// by the slack) bound the cells of all such points.
__device__ __forceinline__ void cell_span(float q, float reach, float lo,
                                          float inv_h, int D, int &c0, int &c1) {
    c0 = cell_axis(__fsub_rn(q, reach), lo, inv_h, D);
    c1 = cell_axis(__fadd_rn(q, reach), lo, inv_h, D);
}

// ---------------------------------------------------------------------------
// Build kernels.
// ---------------------------------------------------------------------------
__global__ void grid_init_kernel(GridHeader *hdr, int D) {
    GridHeader &h = hdr[blockIdx.x];
    if (threadIdx.x < 3) {
        h.kmin[threadIdx.x] = 0xffffffffu;
        h.kmax[threadIdx.x] = 0u;
    }
    if (threadIdx.x == 0) h.D = D;
}

__global__ void grid_bounds_kernel(const float *ref, int N, GridHeader *hdr) {
    const int b = blockIdx.y;
    const float *x = ref + size_t(b) * size_t(N) * 3;
    unsigned mn[3] = {0xffffffffu, 0xffffffffu, 0xffffffffu};
    unsigned mx[3] = {0u, 0u, 0u};
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N;
         j += gridDim.x * blockDim.x) {
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            const unsigned k = order_key(x[size_t(j) * 3 + a]);
            mn[a] = min(mn[a], k);
            mx[a] = max(mx[a], k);
        }
    }
#pragma unroll
    for (int a = 0; a < 3; ++a) {
        mn[a] = __reduce_min_sync(FULL, mn[a]);
        mx[a] = __reduce_max_sync(FULL, mx[a]);
    }
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            atomicMin(&hdr[b].kmin[a], mn[a]);
            atomicMax(&hdr[b].kmax[a], mx[a]);
        }
    }
}

__global__ void grid_finalize_kernel(GridHeader *hdr, int N) {
    GridHeader &h = hdr[blockIdx.x];
    if (threadIdx.x < 3) {
        const int a = threadIdx.x;
        float lo = 0.f, inv_h = 1.f;
        if (N > 0) {
            lo = key_to_float(h.kmin[a]);
            const float hi = key_to_float(h.kmax[a]);
            const float ext = __fsub_rn(hi, lo);
            if (ext > 0.f && isfinite(ext)) {
                const float cell = __fdiv_rn(ext, float(h.D));
                inv_h = cell > 0.f ? __fdiv_rn(1.0f, cell) : 1.0f;
                if (!isfinite(inv_h)) inv_h = 1.0f;
            }
        }
        h.lo[a] = lo;
        h.inv_h[a] = inv_h;
    }
}

__device__ __forceinline__ int point_cell(const GridHeader &h, float x, float y,
                                          float z) {
    const int D = h.D;
    const int cx = cell_axis(x, h.lo[0], h.inv_h[0], D);
    const int cy = cell_axis(y, h.lo[1], h.inv_h[1], D);
    const int cz = cell_axis(z, h.lo[2], h.inv_h[2], D);
    return (cz * D + cy) * D + cx;
}

__global__ void grid_count_kernel(const float *ref, int N, int64_t C,
                                  const GridHeader *hdr, int *count) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const float *p = ref + (size_t(b) * N + j) * 3;
    const int c = point_cell(hdr[b], p[0], p[1], p[2]);
    atomicAdd(&count[size_t(b) * C + c], 1);
}

// Exclusive scan of count[b][0..C) into start[b][0..C], start[b][C] = N; one
// block of 1024 threads per cloud, 4 cells per thread per pass.
__global__ void __launch_bounds__(1024) grid_scan_kernel(const int *count,
                                                         int *start, int64_t C) {
    __shared__ int warp_sums[32];
    __shared__ int carry;
    const int b = blockIdx.x;
    const int *cnt = count + size_t(b) * C;
    int *st = start + size_t(b) * (C + 1);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < C; base += 4096) {
        int v[4], tsum = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t c = base + threadIdx.x * 4 + i;
            v[i] = c < C ? cnt[c] : 0;
            tsum += v[i];
        }
        int incl = tsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(FULL, w, o);
                if (lane >= o) w += t;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        int run = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + (incl - tsum);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t c = base + threadIdx.x * 4 + i;
            if (c < C) st[c] = run;
            run += v[i];
        }
        __syncthreads();
        if (threadIdx.x == 0) carry += warp_sums[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) st[C] = carry;
}

__global__ void grid_scatter_kernel(const float *ref, int N, int64_t C,
                                    const GridHeader *hdr, const int *start,
                                    int *count, float4 *pts) {
    const int b = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= N) return;
    const float *p = ref + (size_t(b) * N + j) * 3;
    const float x = p[0], y = p[1], z = p[2];
    const int c = point_cell(hdr[b], x, y, z);
    const int pos = start[size_t(b) * (C + 1) + c] +
                    atomicSub(&count[size_t(b) * C + c], 1) - 1;
    pts[size_t(b) * N + pos] = make_float4(x, y, z, __int_as_float(j));
}

// ---------------------------------------------------------------------------
// Warp-distributed sorted lists (lane l holds entries l, l + 32, ...).
// ---------------------------------------------------------------------------
// Insert (ks, kj) ordered by (a, b) lexicographically; `less` tells whether
// an entry precedes the candidate.  The list keeps its first 32 * KPL entries.
template <int KPL, class Less>
__device__ __forceinline__ void list_insert(float (&la)[KPL], int (&lb)[KPL],
                                            float ca, int cb, Less less) {
    const int lane = threadIdx.x & 31;
    int pos = 0;
#pragma unroll
    for (int c = 0; c < KPL; ++c) pos += __popc(__ballot_sync(FULL, less(la[c], lb[c])));
#pragma unroll
    for (int c = KPL - 1; c >= 0; --c) {
        float ua = __shfl_up_sync(FULL, la[c], 1);
        int ub = __shfl_up_sync(FULL, lb[c], 1);
        if (c > 0) {
            const float pa = __shfl_sync(FULL, la[c - 1], 31);
            const int pb = __shfl_sync(FULL, lb[c - 1], 31);
            if (lane == 0) {
                ua = pa;
                ub = pb;
            }
        }
        const int e = c * 32 + lane;
        if (e > pos) {
            la[c] = ua;
            lb[c] = ub;
        } else if (e == pos) {
            la[c] = ca;
            lb[c] = cb;
        }
    }
}

template <int KPL>
__device__ __forceinline__ void list_entry(const float (&la)[KPL],
                                           const int (&lb)[KPL], int e,
                                           float &a, int &b) {
    const int ec = e >> 5, el = e & 31;
    float va = la[0];
    int vb = lb[0];
#pragma unroll
    for (int c = 1; c < KPL; ++c)
        if (c == ec) {
            va = la[c];
            vb = lb[c];
        }
    a = __shfl_sync(FULL, va, el);
    b = __shfl_sync(FULL, vb, el);
}

struct QueryArgs {
    const float *query;
    int Q, N, D;
    int64_t C;
    const GridHeader *hdr;
    const int *start;
    const float4 *pts;
    int k;            // kNN: k; Ball Query: K
    float R2;         // Ball Query threshold
    float *out_dist;
    int64_t *out_idx;
};

// ---------------------------------------------------------------------------
// kNN from the grid: one warp per query, cube of half-width R grown a shell
// at a time.
// ---------------------------------------------------------------------------
template <int KPL>
__global__ void __launch_bounds__(256) knn_grid_kernel(const QueryArgs a) {
    const int lane = threadIdx.x & 31;
    const int qi = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int b = blockIdx.y;
    if (qi >= a.Q) return;
    const GridHeader h = a.hdr[b];
    const int D = a.D;
    const float *qp = a.query + (size_t(b) * a.Q + qi) * 3;
    const float qx = qp[0], qy = qp[1], qz = qp[2];
    const int cq[3] = {cell_axis(qx, h.lo[0], h.inv_h[0], D),
                       cell_axis(qy, h.lo[1], h.inv_h[1], D),
                       cell_axis(qz, h.lo[2], h.inv_h[2], D)};
    const int *st = a.start + size_t(b) * (a.C + 1);
    const float4 *pts = a.pts + size_t(b) * a.N;
    const int k = a.k;

    float ls[KPL];
    int lj[KPL];
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
        ls[c] = __int_as_float(0x7f800000);
        lj[c] = INT_MAX;
    }
    float ts = __int_as_float(0x7f800000);
    int tj = INT_MAX;

    auto scan_range = [&](int p0, int p1) {
        for (int base = p0; base < p1; base += 32) {
            const int i = base + lane;
            const bool valid = i < p1;
            float s = 0.f;
            int j = INT_MAX;
            if (valid) {
                const float4 p = pts[i];
                s = sqdist(qx, qy, qz, p.x, p.y, p.z);
                j = __float_as_int(p.w);
            }
            unsigned bal =
                __ballot_sync(FULL, valid && (s < ts || (s == ts && j < tj)));
            while (bal) {
                const int src = __ffs(bal) - 1;
                bal &= bal - 1;
                const float cs = __shfl_sync(FULL, s, src);
                const int cj = __shfl_sync(FULL, j, src);
                if (cs < ts || (cs == ts && cj < tj)) {
                    list_insert<KPL>(ls, lj, cs, cj, [&](float ea, int eb) {
                        return ea < cs || (ea == cs && eb < cj);
                    });
                    list_entry<KPL>(ls, lj, k - 1, ts, tj);
                }
            }
        }
    };
    auto scan_row = [&](int z, int y, int x0, int x1) {
        const int64_t c0 = (int64_t(z) * D + y) * D + x0;
        scan_range(st[c0], st[c0 + (x1 - x0) + 1]);
    };

    const float slack = query_slack(qx, qy, qz);
    const float qf[3] = {qx, qy, qz};

    for (int R = 0; R <= D; ++R) {
        // the shell of half-width R: rows with |dz| == R or |dy| == R in
        // full, the others only at x = cx - R and cx + R
        for (int dz = -R; dz <= R; ++dz) {
            const int z = cq[2] + dz;
            if (z < 0 || z >= D) continue;
            for (int dy = -R; dy <= R; ++dy) {
                const int y = cq[1] + dy;
                if (y < 0 || y >= D) continue;
                if (dz == -R || dz == R || dy == -R || dy == R) {
                    scan_row(z, y, max(cq[0] - R, 0), min(cq[0] + R, D - 1));
                } else if (R > 0) {
                    if (cq[0] - R >= 0) scan_row(z, y, cq[0] - R, cq[0] - R);
                    if (cq[0] + R < D) scan_row(z, y, cq[0] + R, cq[0] + R);
                }
            }
        }
        // done once the cube holds every cell that can contain a point with
        // s32 <= tau (the current k-th squared distance), or all cells
        bool covered = true;
        const float reach =
            tj == INT_MAX ? __int_as_float(0x7f800000)
                          : __fsqrt_rn(ts) * (1.0f + 1e-5f) + slack;
#pragma unroll
        for (int ax = 0; ax < 3; ++ax) {
            int c0, c1;
            cell_span(qf[ax], reach, h.lo[ax], h.inv_h[ax], D, c0, c1);
            covered = covered && c0 >= cq[ax] - R && c1 <= cq[ax] + R;
        }
        if (covered) break;
    }

    const size_t row = size_t(b) * a.Q + qi;
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
        const int e = c * 32 + lane;
        if (e < k) {
            a.out_idx[row * k + e] = lj[c];
            a.out_dist[row * k + e] = __fsqrt_rn(ls[c]);
        }
    }
}

// ---------------------------------------------------------------------------
// Ball Query from the grid: one warp per query; the cells that can hold a
// hit; the K smallest indices among the hits.
// ---------------------------------------------------------------------------
template <int KPL>
__global__ void __launch_bounds__(256) bq_grid_kernel(const QueryArgs a,
                                                       float r32) {
    const int lane = threadIdx.x & 31;
    const int qi = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int b = blockIdx.y;
    if (qi >= a.Q) return;
    const int K = a.k;
    const size_t row = size_t(b) * a.Q + qi;
    float ls[KPL];
    int lj[KPL];
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
        ls[c] = 0.f;
        lj[c] = INT_MAX;
    }
    int hits = 0;
    if (a.N > 0) {
        const GridHeader h = a.hdr[b];
        const int D = a.D;
        const float *qp = a.query + row * 3;
        const float qx = qp[0], qy = qp[1], qz = qp[2];
        const float qf[3] = {qx, qy, qz};
        const int *st = a.start + size_t(b) * (a.C + 1);
        const float4 *pts = a.pts + size_t(b) * a.N;
        // every point with s32 < fl(r^2) lies in these cells
        const float reach = r32 * (1.0f + 1e-5f) + query_slack(qx, qy, qz);
        int lo_c[3], hi_c[3];
#pragma unroll
        for (int ax = 0; ax < 3; ++ax)
            cell_span(qf[ax], reach, h.lo[ax], h.inv_h[ax], D, lo_c[ax], hi_c[ax]);
        int tj = INT_MAX;  // K-th smallest index among the hits so far
        for (int z = lo_c[2]; z <= hi_c[2]; ++z) {
            for (int y = lo_c[1]; y <= hi_c[1]; ++y) {
                const int64_t c0 = (int64_t(z) * D + y) * D + lo_c[0];
                const int p0 = st[c0];
                const int p1 = st[c0 + (hi_c[0] - lo_c[0]) + 1];
                for (int base = p0; base < p1; base += 32) {
                    const int i = base + lane;
                    const bool valid = i < p1;
                    float s = 0.f;
                    int j = INT_MAX;
                    if (valid) {
                        const float4 p = pts[i];
                        s = sqdist(qx, qy, qz, p.x, p.y, p.z);
                        j = __float_as_int(p.w);
                    }
                    unsigned bal = __ballot_sync(FULL, valid && s < a.R2 && j < tj);
                    while (bal) {
                        const int src = __ffs(bal) - 1;
                        bal &= bal - 1;
                        const float cs = __shfl_sync(FULL, s, src);
                        const int cj = __shfl_sync(FULL, j, src);
                        if (cj < tj) {
                            list_insert<KPL>(ls, lj, cs, cj, [&](float, int eb) {
                                return eb < cj;
                            });
                            ++hits;
                            if (hits >= K) {
                                float dummy;
                                list_entry<KPL>(ls, lj, K - 1, dummy, tj);
                            }
                        }
                    }
                }
            }
        }
    }
    const int n = min(hits, K);
#pragma unroll
    for (int c = 0; c < KPL; ++c) {
        const int e = c * 32 + lane;
        if (e < K) {
            a.out_idx[row * K + e] = e < n ? int64_t(lj[c]) : int64_t(-1);
            a.out_dist[row * K + e] = e < n ? ls[c] : 0.0f;
        }
    }
}

}  // namespace
}  // namespace pcn

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
namespace {

int bad(int code, const char *msg) { return pcn::api_fail(code, msg); }

bool sizes_ok(int64_t B, int64_t N) {
    return B >= 0 && N >= 0 && B <= 65535 && N <= 2147483647 &&
           B * N <= (int64_t(1) << 40);
}

}  // namespace

extern "C" size_t pc_grid_bytes(int64_t B, int64_t N) {
    if (!sizes_ok(B, N)) return 0;
    return pcn::grid_geometry(B, N).total;
}

extern "C" int pc_grid_build(const float *ref, int64_t B, int64_t N,
                             void *grid, size_t grid_bytes, void *stream) {
    if (!sizes_ok(B, N))
        return bad(PC_ERR_INVALID_ARGUMENT, "grid_build: bad B or N");
    if (B == 0) return PC_OK;
    const pcn::GridGeometry g = pcn::grid_geometry(B, N);
    if (grid_bytes < g.total) {
        char m[160];
        std::snprintf(m, sizeof(m), "grid_build: grid of %zu bytes, need %zu",
                      grid_bytes, g.total);
        return bad(PC_ERR_INVALID_ARGUMENT, m);
    }
    const pcn::DeviceInfo *dev = nullptr;
    int rc = pcn::api_current_device(&dev);
    if (rc != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(grid, dev->device, 256, "grid")) != PC_OK) return rc;
    if (N > 0 && (rc = pcn::api_check_ptr(ref, dev->device, 4, "ref")) != PC_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *base = static_cast<unsigned char *>(grid);
    auto *hdr = reinterpret_cast<pcn::GridHeader *>(base + g.off_header);
    int *start = reinterpret_cast<int *>(base + g.off_start);
    int *count = reinterpret_cast<int *>(base + g.off_count);
    float4 *pts = reinterpret_cast<float4 *>(base + g.off_pts);
    cudaError_t e = cudaMemsetAsync(count, 0, size_t(B) * size_t(g.C) * 4, st);
    if (e == cudaSuccess) {
        pcn::grid_init_kernel<<<unsigned(B), 32, 0, st>>>(hdr, g.D);
        if (N > 0) {
            const unsigned nb = unsigned(std::min<int64_t>((N + 255) / 256, 256));
            pcn::grid_bounds_kernel<<<dim3(nb, unsigned(B)), 256, 0, st>>>(ref, int(N), hdr);
        }
        pcn::grid_finalize_kernel<<<unsigned(B), 32, 0, st>>>(hdr, int(N));
        if (N > 0) {
            const dim3 pg(unsigned((N + 255) / 256), unsigned(B));
            pcn::grid_count_kernel<<<pg, 256, 0, st>>>(ref, int(N), g.C, hdr, count);
            pcn::grid_scan_kernel<<<unsigned(B), 1024, 0, st>>>(count, start, g.C);
            pcn::grid_scatter_kernel<<<pg, 256, 0, st>>>(ref, int(N), g.C, hdr,
                                                         start, count, pts);
        } else {
            pcn::grid_scan_kernel<<<unsigned(B), 1024, 0, st>>>(count, start, g.C);
        }
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) {
        char m[200];
        std::snprintf(m, sizeof(m), "grid_build: %s", cudaGetErrorString(e));
        return bad(PC_ERR_CUDA, m);
    }
    return PC_OK;
}

namespace {

int query_common(const float *query, int64_t B, int64_t Q, const void *grid,
                 int64_t N, void *out_a, void *out_b, const pcn::DeviceInfo **dev) {
    int rc = pcn::api_current_device(dev);
    if (rc != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(query, (*dev)->device, 4, "query")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(grid, (*dev)->device, 256, "grid")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(out_a, (*dev)->device, 4, "out_dist")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(out_b, (*dev)->device, 8, "out_idx")) != PC_OK) return rc;
    (void)B;
    (void)Q;
    (void)N;
    return PC_OK;
}

pcn::QueryArgs make_args(const float *query, int64_t B, int64_t Q,
                         const void *grid, int64_t N, int k, float *out_dist,
                         int64_t *out_idx) {
    const pcn::GridView v = pcn::grid_view(grid, B, N);
    pcn::QueryArgs a{};
    a.query = query;
    a.Q = int(Q);
    a.N = int(N);
    a.D = v.D;
    a.C = v.C;
    a.hdr = v.hdr;
    a.start = v.start;
    a.pts = v.pts;
    a.k = k;
    a.out_dist = out_dist;
    a.out_idx = out_idx;
    return a;
}

}  // namespace

extern "C" int pc_knn_grid(const float *query, int64_t B, int64_t Q,
                           const void *grid, int64_t N, int64_t k,
                           float *out_dist, int64_t *out_idx, void *stream) {
    if (!sizes_ok(B, N) || Q < 0 || Q > 2147483647)
        return bad(PC_ERR_INVALID_ARGUMENT, "knn_grid: bad B, Q or N");
    if (k < 1 || k > N)
        return bad(PC_ERR_INVALID_ARGUMENT, "knn_grid: need 1 <= k <= N");
    if (k > pcn::kMaxKGrid)
        return bad(PC_ERR_UNSUPPORTED, "knn_grid: k above 256");
    if (B == 0 || Q == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    int rc = query_common(query, B, Q, grid, N, out_dist, out_idx, &dev);
    if (rc != PC_OK) return rc;
    const pcn::QueryArgs a = make_args(query, B, Q, grid, N, int(k), out_dist, out_idx);
    const dim3 g(unsigned((Q + 7) / 8), unsigned(B));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (k <= 32) pcn::knn_grid_kernel<1><<<g, 256, 0, st>>>(a);
    else if (k <= 64) pcn::knn_grid_kernel<2><<<g, 256, 0, st>>>(a);
    else if (k <= 128) pcn::knn_grid_kernel<4><<<g, 256, 0, st>>>(a);
    else pcn::knn_grid_kernel<8><<<g, 256, 0, st>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return bad(PC_ERR_CUDA, cudaGetErrorString(e));
    return PC_OK;
}

extern "C" int pc_ball_query_grid(const float *query, int64_t B, int64_t Q,
                                  const void *grid, int64_t N, double radius,
                                  int64_t K, float *out_dist2, int64_t *out_idx,
                                  void *stream) {
    if (!sizes_ok(B, N) || Q < 0 || Q > 2147483647)
        return bad(PC_ERR_INVALID_ARGUMENT, "ball_query_grid: bad B, Q or N");
    if (!std::isfinite(radius) || !(radius > 0.0))
        return bad(PC_ERR_INVALID_ARGUMENT, "ball_query_grid: radius must be finite and > 0");
    if (K < 1) return bad(PC_ERR_INVALID_ARGUMENT, "ball_query_grid: need K >= 1");
    if (K > pcn::kMaxKGrid)
        return bad(PC_ERR_UNSUPPORTED, "ball_query_grid: K above 256");
    if (B == 0 || Q == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    int rc = query_common(query, B, Q, grid, N, out_dist2, out_idx, &dev);
    if (rc != PC_OK) return rc;
    pcn::QueryArgs a = make_args(query, B, Q, grid, N, int(K), out_dist2, out_idx);
    const float r32 = static_cast<float>(radius);
    a.R2 = r32 * r32;  // fl32(fl32(r) * fl32(r))
    const dim3 g(unsigned((Q + 7) / 8), unsigned(B));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K <= 32) pcn::bq_grid_kernel<1><<<g, 256, 0, st>>>(a, r32);
    else if (K <= 64) pcn::bq_grid_kernel<2><<<g, 256, 0, st>>>(a, r32);
    else if (K <= 128) pcn::bq_grid_kernel<4><<<g, 256, 0, st>>>(a, r32);
    else pcn::bq_grid_kernel<8><<<g, 256, 0, st>>>(a, r32);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return bad(PC_ERR_CUDA, cudaGetErrorString(e));
    return PC_OK;
}
