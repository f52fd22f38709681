// pc_interp.cu -- PointNet++ feature propagation (three_interpolate forward
// and backward) and the neighbor-coordinate gather on sm_103a.
//
// three_interpolate (mps-pointops project page, "Quick start"; "Roadmap",
// Phase 2: externally computed weights, gradients accumulated into the input
// features):
//   out[b,c,i] = sum_{t<3} w[b,i,t] f[b,c,idx[b,i,t]]     f [B,C,M], out [B,C,n]
//   grad_f[b,c,m] += w[b,i,t] g[b,c,i]  for every idx[b,i,t] = m.
// Forward: float32, products and sums rounded separately in the order
// ((w0 f0 + w1 f1) + w2 f2), so the result is bit-identical to the oracle's.
// Backward (M, n <= 16384): deterministic and bit-exact with the oracle -- each
// grad_f[b, c, m] is summed from 0 in increasing (i, t) order, each product
// and addition rounded.  Per cloud a CSR of the entries (i, t) of every m,
// in increasing entry order, is built once (count, scan, fill, then a sort of
// each short segment by entry), then
// one thread per (b, m) sums its list for a chunk of channels whose
// grad_out rows are staged in shared memory.  Larger sizes: float32 atomic adds
// (order unspecified, as the pages allow for accumulated gradients).
// idx = -1 is padding (reads 0, adds nothing); any other index outside
// [0, M) sets PC_ERR_INVALID_ARGUMENT in the device status word and is
// treated as padding.
//
// Staged kernels (used when a chunk of channels of one cloud fits in shared
// memory, M <= 16384): a block owns (cloud b, channels c0 .. c0 + CC):
//   forward  -- copies f[b, c0.., :] into shared memory (coalesced), then for
//               a range of points i reads the three (index, weight) pairs once
//               and writes out[b, c, i] for its CC channels (coalesced along
//               i), gathering from shared memory;
// Otherwise the direct kernel gathers from global memory (L2) with one thread
// per point.
//
// gather_points (project page, "PyTorch3D-style Ball Query": return_nn gives
// the neighbor coordinates, zeros where idx = -1):
//   out[b,q,t,:] = x[b, idx[b,q,t], :].
#include "pointcloud.h"
#include "pc_device.cuh"
#include "pc_internal.h"

#include <algorithm>
#include <cstdio>

namespace pcn {
namespace {

constexpr int INTERP_THREADS = 128;
constexpr int INTERP_CCHUNK = 16;  // channels per block

// Load the three (index, weight) pairs of point i; bad indices become padding
// and raise the status word.
__device__ __forceinline__ void load_triplet(const int64_t *idx,
                                             const float *w, size_t base,
                                             int M, int (&m)[3], float (&wt)[3],
                                             int *status) {
#pragma unroll
    for (int t = 0; t < 3; ++t) {
        const int64_t v = idx[base + t];
        wt[t] = w[base + t];
        if (v == -1) {
            m[t] = -1;
        } else if (v < 0 || v >= M) {
            m[t] = -1;
            raise_status(status, PC_ERR_INVALID_ARGUMENT);
        } else {
            m[t] = static_cast<int>(v);
        }
    }
}

__global__ void __launch_bounds__(INTERP_THREADS)
three_interpolate_kernel(const float *__restrict__ f,
                         const int64_t *__restrict__ idx,
                         const float *__restrict__ w, int C, int M, int n,
                         float *__restrict__ out, int *status) {
    const int i = blockIdx.x * INTERP_THREADS + threadIdx.x;
    if (i >= n) return;
    const int b = blockIdx.z;
    const int c0 = blockIdx.y * INTERP_CCHUNK;
    const int c1 = min(C, c0 + INTERP_CCHUNK);
    int m[3];
    float wt[3];
    load_triplet(idx, w, (size_t(b) * n + i) * 3, M, m, wt, status);
#pragma unroll 4
    for (int c = c0; c < c1; ++c) {
        const float *fr = f + (size_t(b) * C + c) * size_t(M);
        const float v0 = m[0] >= 0 ? __ldg(fr + m[0]) : 0.0f;
        const float v1 = m[1] >= 0 ? __ldg(fr + m[1]) : 0.0f;
        const float v2 = m[2] >= 0 ? __ldg(fr + m[2]) : 0.0f;
        const float s01 = __fadd_rn(__fmul_rn(wt[0], v0), __fmul_rn(wt[1], v1));
        out[(size_t(b) * C + c) * size_t(n) + i] = __fadd_rn(s01, __fmul_rn(wt[2], v2));
    }
}

__global__ void __launch_bounds__(INTERP_THREADS)
three_interpolate_backward_kernel(const float *__restrict__ g,
                                  const int64_t *__restrict__ idx,
                                  const float *__restrict__ w, int C, int M,
                                  int n, float *grad_f, int *status) {
    const int i = blockIdx.x * INTERP_THREADS + threadIdx.x;
    if (i >= n) return;
    const int b = blockIdx.z;
    const int c0 = blockIdx.y * INTERP_CCHUNK;
    const int c1 = min(C, c0 + INTERP_CCHUNK);
    int m[3];
    float wt[3];
    load_triplet(idx, w, (size_t(b) * n + i) * 3, M, m, wt, status);
#pragma unroll 4
    for (int c = c0; c < c1; ++c) {
        const float gv = __ldg(g + (size_t(b) * C + c) * size_t(n) + i);
        float *gr = grad_f + (size_t(b) * C + c) * size_t(M);
#pragma unroll
        for (int t = 0; t < 3; ++t)
            if (m[t] >= 0) atomicAdd(gr + m[t], __fmul_rn(wt[t], gv));
    }
}

// --- staged (shared-memory) kernels -------------------------------------------
constexpr int STG_THREADS = 256;
constexpr int STG_SMEM_FLOATS = 16384;   // 64 KB of features per block
constexpr int STG_POINTS = 1024;         // points per forward block

__global__ void __launch_bounds__(STG_THREADS)
three_interpolate_staged_kernel(const float *__restrict__ f,
                                const int64_t *__restrict__ idx,
                                const float *__restrict__ w, int C, int M, int n,
                                int CC, float *__restrict__ out, int *status) {
    extern __shared__ float tile[];  // [CC][M]
    const int b = blockIdx.z;
    const int c0 = blockIdx.y * CC;
    const int cc = min(CC, C - c0);
    const float *fb = f + (size_t(b) * C + c0) * size_t(M);
    const int ne = cc * M;
    if ((reinterpret_cast<uintptr_t>(fb) & 15) == 0) {  // 128-bit loads
        const float4 *f4 = reinterpret_cast<const float4 *>(fb);
        float4 *t4 = reinterpret_cast<float4 *>(tile);
        for (int e = threadIdx.x; e < ne / 4; e += STG_THREADS) t4[e] = __ldg(f4 + e);
        for (int e = (ne & ~3) + threadIdx.x; e < ne; e += STG_THREADS) tile[e] = __ldg(fb + e);
    } else {
        for (int e = threadIdx.x; e < ne; e += STG_THREADS) tile[e] = __ldg(fb + e);
    }
    // the (index, weight) triplets of this thread's points, all loads in
    // flight at once while the features are staged
    constexpr int PPT = STG_POINTS / STG_THREADS;
    const int i0 = blockIdx.x * STG_POINTS + threadIdx.x;
    int m[PPT][3];
    float wt[PPT][3];
#pragma unroll
    for (int p = 0; p < PPT; ++p) {
        const int i = i0 + p * STG_THREADS;
        if (i < n) {
            load_triplet(idx, w, (size_t(b) * n + i) * 3, M, m[p], wt[p], status);
        } else {
#pragma unroll
            for (int t = 0; t < 3; ++t) {
                m[p][t] = -1;
                wt[p][t] = 0.0f;
            }
        }
    }
    __syncthreads();
    for (int c = 0; c < cc; ++c) {
        const float *tr = tile + c * M;
        float *oc = out + (size_t(b) * C + c0 + c) * size_t(n);
#pragma unroll
        for (int p = 0; p < PPT; ++p) {
            const int i = i0 + p * STG_THREADS;
            const float v0 = m[p][0] >= 0 ? tr[m[p][0]] : 0.0f;
            const float v1 = m[p][1] >= 0 ? tr[m[p][1]] : 0.0f;
            const float v2 = m[p][2] >= 0 ? tr[m[p][2]] : 0.0f;
            const float s01 =
                __fadd_rn(__fmul_rn(wt[p][0], v0), __fmul_rn(wt[p][1], v1));
            if (i < n) oc[i] = __fadd_rn(s01, __fmul_rn(wt[p][2], v2));
        }
    }
}

// --- deterministic backward: per-cloud CSR, then ordered sums ---------------
constexpr int CSR_THREADS = 1024;

// One block per cloud: counts of every m (shared-memory atomics), exclusive
// scan into start[b][0..M], then every entry e = 3 i + t is placed in its m's
// segment at a cursor taken with a shared-memory atomic, as the pair
// (e, weight) -- the order inside a segment is fixed afterwards by
// interp_sort_kernel.
__global__ void __launch_bounds__(CSR_THREADS)
interp_csr_kernel(const int64_t *__restrict__ idx, const float *__restrict__ w,
                  int n, int M, int *__restrict__ start, int2 *__restrict__ list,
                  int *status) {
    extern __shared__ int cnt[];  // [M] counts then cursors, [32] warp sums
    int *wsum = cnt + M;
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = 3 * n;
    const int64_t *ib = idx + size_t(b) * E;
    for (int m = tid; m < M; m += CSR_THREADS) cnt[m] = 0;
    __syncthreads();
    for (int e = tid; e < E; e += CSR_THREADS) {
        const int64_t v = ib[e];
        if (v >= 0 && v < M)
            atomicAdd(&cnt[v], 1);
        else if (v != -1)
            raise_status(status, PC_ERR_INVALID_ARGUMENT);
    }
    __syncthreads();
    // exclusive scan: thread tid owns [tid * ch, (tid + 1) * ch)
    const int ch = (M + CSR_THREADS - 1) / CSR_THREADS;
    const int m0 = min(M, tid * ch), m1 = min(M, m0 + ch);
    int local = 0;
    for (int m = m0; m < m1; ++m) local += cnt[m];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += t;
        }
        wsum[lane] = x;
    }
    __syncthreads();
    int run = (warp > 0 ? wsum[warp - 1] : 0) + incl - local;
    int *sb = start + size_t(b) * (M + 1);
    for (int m = m0; m < m1; ++m) {
        const int c = cnt[m];
        cnt[m] = run;  // becomes the cursor of m
        sb[m] = run;
        run += c;
    }
    if (tid == CSR_THREADS - 1) sb[M] = wsum[31];
    __syncthreads();
    int2 *lb = list + size_t(b) * E;
    const float *wb = w + size_t(b) * E;
    for (int e = tid; e < E; e += CSR_THREADS) {
        const int64_t v = ib[e];
        if (v >= 0 && v < M) {
            const int p = atomicAdd(&cnt[v], 1);
            lb[p] = make_int2(e, __float_as_int(wb[e]));
        }
    }
}

// One thread per (b, m): insertion sort of m's segment by entry e (segments
// hold ~3n/M entries), so the sums run in increasing (i, t) order.  A
// segment of up to SORT_LOCAL entries is sorted in the thread's slice of
// shared memory (one global read and write per entry); longer ones in place.
constexpr int SORT_THREADS = 128;
constexpr int SORT_LOCAL = 32;
__global__ void __launch_bounds__(SORT_THREADS)
interp_sort_kernel(const int *__restrict__ start, int2 *__restrict__ list, int B, int M,
                   int n) {
    __shared__ int2 buf[SORT_THREADS * (SORT_LOCAL + 1)];
    const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= int64_t(B) * M) return;
    const int b = int(t / M), m = int(t % M);
    const int *sb = start + size_t(b) * (M + 1);
    int2 *lb = list + size_t(b) * 3 * n;
    const int p0 = sb[m], p1 = sb[m + 1];
    const int L = p1 - p0;
    if (L <= SORT_LOCAL) {
        int2 *mine = buf + threadIdx.x * (SORT_LOCAL + 1);
        for (int u = 0; u < L; ++u) mine[u] = lb[p0 + u];
        for (int p = 1; p < L; ++p) {
            const int2 v = mine[p];
            int q = p - 1;
            while (q >= 0 && mine[q].x > v.x) {
                mine[q + 1] = mine[q];
                --q;
            }
            mine[q + 1] = v;
        }
        for (int u = 0; u < L; ++u) lb[p0 + u] = mine[u];
        return;
    }
    for (int p = p0 + 1; p < p1; ++p) {
        const int2 v = lb[p];
        int q = p - 1;
        while (q >= p0 && lb[q].x > v.x) {
            lb[q + 1] = lb[q];
            --q;
        }
        lb[q + 1] = v;
    }
}

// A block owns (cloud b, channels c0 .. c0 + 4): it stages grad_out[b, c, :]
// for its channels in shared memory point-major (the 4 channels of a point
// are one 16-byte word), then each thread, for its m, walks the sorted
// entries of m and accumulates w * g for the 4 channels:
//   grad_f[b, c, m] = sum over e of w[b, e] * g[b, c, e / 3]
// (each product and sum rounded, from 0).
constexpr int GATH_THREADS = 256;
constexpr int GATH_SMEM_FLOATS = 32768;  // 128 KB of grad_out per block (n <= 8192)
constexpr int GATH_CC = 4;

__global__ void __launch_bounds__(GATH_THREADS)
interp_gather_kernel(const float *__restrict__ g, const int *__restrict__ start,
                     const int2 *__restrict__ list, int C, int M, int n,
                     float *__restrict__ grad_f) {
    extern __shared__ float4 gt4[];  // [n]: channels c0 .. c0 + 3 of point i
    const int b = blockIdx.y;
    const int c0 = blockIdx.x * GATH_CC;
    const int cc = min(GATH_CC, C - c0);
    const float *gb = g + (size_t(b) * C + c0) * size_t(n);
    // point-major staging: the 4 channels of point i as one 16-byte word
    for (int i = threadIdx.x; i < n; i += GATH_THREADS) {
        float v[GATH_CC];
#pragma unroll
        for (int c = 0; c < GATH_CC; ++c) v[c] = c < cc ? __ldg(gb + size_t(c) * n + i) : 0.0f;
        gt4[i] = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
    const int *sb = start + size_t(b) * (M + 1);
    const int2 *lb = list + size_t(b) * 3 * n;
    for (int m = threadIdx.x; m < M; m += GATH_THREADS) {
        const int p0 = sb[m], p1 = sb[m + 1];
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        for (int pc = p0; pc < p1; pc += 16) {
            int2 v[16];  // the next 16 entries, loaded before any is used
#pragma unroll
            for (int u = 0; u < 16; ++u)
                v[u] = pc + u < p1 ? __ldg(lb + pc + u) : make_int2(0, 0);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (pc + u >= p1) break;
                const float wv = __int_as_float(v[u].y);
                const float4 gv = gt4[v[u].x / 3];
                a0 = __fadd_rn(a0, __fmul_rn(wv, gv.x));
                a1 = __fadd_rn(a1, __fmul_rn(wv, gv.y));
                a2 = __fadd_rn(a2, __fmul_rn(wv, gv.z));
                a3 = __fadd_rn(a3, __fmul_rn(wv, gv.w));
            }
        }
        float *out = grad_f + (size_t(b) * C + c0) * size_t(M) + m;
        out[0] = a0;
        if (cc > 1) out[size_t(M)] = a1;
        if (cc > 2) out[2 * size_t(M)] = a2;
        if (cc > 3) out[3 * size_t(M)] = a3;
    }
}

__global__ void gather_points_kernel(const float *__restrict__ x, int N,
                                     const int64_t *__restrict__ idx,
                                     int64_t QK, int64_t total,
                                     float *__restrict__ out, int *status) {
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t b = e / QK;
        const int64_t j = idx[e];
        float px = 0.f, py = 0.f, pz = 0.f;
        if (j >= 0 && j < N) {
            const float *p = x + (size_t(b) * N + size_t(j)) * 3;
            px = p[0];
            py = p[1];
            pz = p[2];
        } else if (j != -1) {
            raise_status(status, PC_ERR_INVALID_ARGUMENT);
        }
        out[e * 3 + 0] = px;
        out[e * 3 + 1] = py;
        out[e * 3 + 2] = pz;
    }
}

}  // namespace
}  // namespace pcn

namespace {

constexpr int64_t kMaxInt = 2147483647;

int cuda_err(cudaError_t e, const char *what) {
    char m[200];
    std::snprintf(m, sizeof(m), "%s: %s", what, cudaGetErrorString(e));
    return pcn::api_fail(PC_ERR_CUDA, m);
}

// Sizes of a [B, C, n] / [B, C, M] problem: non-negative, within 32-bit
// point indexing and 2^40 elements per tensor.
int interp_sizes(const char *what, int64_t B, int64_t C, int64_t M, int64_t n) {
    char m[200];
    if (B < 0 || C < 0 || M < 0 || n < 0) {
        std::snprintf(m, sizeof(m), "%s: negative size", what);
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, m);
    }
    const int64_t lim = int64_t(1) << 40;
    const int64_t longest = std::max<int64_t>(std::max<int64_t>(M, n), 1);
    if (B > 65535 || C > int64_t(65535) * 16 || M > kMaxInt || n > kMaxInt ||
        B * C > lim / longest) {
        std::snprintf(m, sizeof(m), "%s: sizes beyond the supported range", what);
        return pcn::api_fail(PC_ERR_UNSUPPORTED, m);
    }
    return PC_OK;
}

}  // namespace

extern "C" int pc_three_interpolate(const float *features, int64_t B,
                                    int64_t C, int64_t M, const int64_t *idx,
                                    const float *weight, int64_t n, float *out,
                                    void *stream) {
    int rc = interp_sizes("three_interpolate", B, C, M, n);
    if (rc != PC_OK) return rc;
    if (B == 0 || C == 0 || n == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    if ((rc = pcn::api_current_device(&dev)) != PC_OK) return rc;
    const int d = dev->device;
    if (M > 0 && (rc = pcn::api_check_ptr(features, d, 4, "features")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(idx, d, 8, "idx")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(weight, d, 4, "weight")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(out, d, 4, "out")) != PC_OK) return rc;
    cudaError_t e;
    if (M > 0 && M <= pcn::STG_SMEM_FLOATS) {
        const int CC = int(std::min<int64_t>(C, pcn::STG_SMEM_FLOATS / M));
        const size_t smem = size_t(CC) * size_t(M) * sizeof(float);
        e = cudaFuncSetAttribute(pcn::three_interpolate_staged_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e == cudaSuccess) {
            const dim3 grid(unsigned((n + pcn::STG_POINTS - 1) / pcn::STG_POINTS),
                            unsigned((C + CC - 1) / CC), unsigned(B));
            pcn::three_interpolate_staged_kernel<<<grid, pcn::STG_THREADS, smem,
                                                   static_cast<cudaStream_t>(stream)>>>(
                features, idx, weight, int(C), int(M), int(n), CC, out,
                dev->status_word);
            e = cudaGetLastError();
        }
    } else {
        const dim3 grid(unsigned((n + pcn::INTERP_THREADS - 1) / pcn::INTERP_THREADS),
                        unsigned((C + pcn::INTERP_CCHUNK - 1) / pcn::INTERP_CCHUNK),
                        unsigned(B));
        pcn::three_interpolate_kernel<<<grid, pcn::INTERP_THREADS, 0,
                                        static_cast<cudaStream_t>(stream)>>>(
            features, idx, weight, int(C), int(M), int(n), out, dev->status_word);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? PC_OK : cuda_err(e, "three_interpolate: launch");
}

extern "C" int pc_three_interpolate_backward(const float *grad_out, int64_t B,
                                             int64_t C, int64_t n,
                                             const int64_t *idx,
                                             const float *weight, int64_t M,
                                             float *grad_features,
                                             void *stream) {
    int rc = interp_sizes("three_interpolate_backward", B, C, M, n);
    if (rc != PC_OK) return rc;
    if (B == 0 || C == 0 || M == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    if ((rc = pcn::api_current_device(&dev)) != PC_OK) return rc;
    const int d = dev->device;
    if ((rc = pcn::api_check_ptr(grad_features, d, 4, "grad_features")) != PC_OK)
        return rc;
    if (n > 0) {
        if ((rc = pcn::api_check_ptr(grad_out, d, 4, "grad_out")) != PC_OK) return rc;
        if ((rc = pcn::api_check_ptr(idx, d, 8, "idx")) != PC_OK) return rc;
        if ((rc = pcn::api_check_ptr(weight, d, 4, "weight")) != PC_OK) return rc;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (M <= pcn::STG_SMEM_FLOATS && n <= pcn::GATH_SMEM_FLOATS / pcn::GATH_CC) {
        // deterministic path: stream-ordered scratch for the per-cloud CSR
        const size_t E = size_t(3) * size_t(n);
        const size_t start_bytes = (size_t(B) * (size_t(M) + 1) * sizeof(int) + 15) & ~size_t(15);
        const size_t bytes = start_bytes + size_t(B) * E * sizeof(int2);
        void *scratch = nullptr;
        cudaError_t e = pcn::scratch_alloc(*dev, &scratch, bytes, st);
        if (e != cudaSuccess) return cuda_err(e, "three_interpolate_backward: scratch");
        int *start = static_cast<int *>(scratch);
        int2 *list = reinterpret_cast<int2 *>(static_cast<char *>(scratch) + start_bytes);
        const size_t csr_smem = (size_t(M) + 32) * sizeof(int);
        e = cudaFuncSetAttribute(pcn::interp_csr_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(csr_smem));
        if (e == cudaSuccess) {
            pcn::interp_csr_kernel<<<unsigned(B), pcn::CSR_THREADS, csr_smem, st>>>(
                idx, weight, int(n), int(M), start, list, dev->status_word);
            e = cudaGetLastError();
        }
        if (e == cudaSuccess) {
            const int64_t segs = B * M;
            pcn::interp_sort_kernel<<<unsigned((segs + pcn::SORT_THREADS - 1) /
                                               pcn::SORT_THREADS),
                                      pcn::SORT_THREADS, 0, st>>>(
                start, list, int(B), int(M), int(n));
            e = cudaGetLastError();
        }
        const size_t g_smem = size_t(pcn::GATH_CC) * size_t(std::max<int64_t>(n, 1)) *
                              sizeof(float);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(pcn::interp_gather_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(g_smem));
        if (e == cudaSuccess) {
            const dim3 grid(unsigned((C + pcn::GATH_CC - 1) / pcn::GATH_CC), unsigned(B));
            pcn::interp_gather_kernel<<<grid, pcn::GATH_THREADS, g_smem, st>>>(
                grad_out, start, list, int(C), int(M), int(n), grad_features);
            e = cudaGetLastError();
        }
        const cudaError_t ef = pcn::scratch_free(scratch, st);
        if (e == cudaSuccess) e = ef;
        return e == cudaSuccess ? PC_OK : cuda_err(e, "three_interpolate_backward");
    }
    cudaError_t e = cudaMemsetAsync(grad_features, 0,
                                    size_t(B) * size_t(C) * size_t(M) * sizeof(float), st);
    if (e == cudaSuccess && n > 0) {
        const dim3 grid(unsigned((n + pcn::INTERP_THREADS - 1) / pcn::INTERP_THREADS),
                        unsigned((C + pcn::INTERP_CCHUNK - 1) / pcn::INTERP_CCHUNK),
                        unsigned(B));
        pcn::three_interpolate_backward_kernel<<<grid, pcn::INTERP_THREADS, 0, st>>>(
            grad_out, idx, weight, int(C), int(M), int(n), grad_features,
            dev->status_word);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? PC_OK : cuda_err(e, "three_interpolate_backward");
}

extern "C" int pc_gather_points(const float *xyz, int64_t B, int64_t N,
                                const int64_t *idx, int64_t Q, int64_t K,
                                float *out, void *stream) {
    if (B < 0 || N < 0 || Q < 0 || K < 0)
        return pcn::api_fail(PC_ERR_INVALID_ARGUMENT, "gather_points: negative size");
    if (N > kMaxInt || B > 65535 || (Q > 0 && K > (int64_t(1) << 40) / Q) ||
        (Q * K > 0 && B > (int64_t(1) << 40) / (Q * K)))
        return pcn::api_fail(PC_ERR_UNSUPPORTED, "gather_points: sizes beyond the supported range");
    const int64_t total = B * Q * K;
    if (total == 0) return PC_OK;
    const pcn::DeviceInfo *dev = nullptr;
    int rc = pcn::api_current_device(&dev);
    if (rc != PC_OK) return rc;
    const int d = dev->device;
    if (N > 0 && (rc = pcn::api_check_ptr(xyz, d, 4, "xyz")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(idx, d, 8, "idx")) != PC_OK) return rc;
    if ((rc = pcn::api_check_ptr(out, d, 4, "out")) != PC_OK) return rc;
    const int64_t blocks = (total + 255) / 256;
    const unsigned grid = unsigned(blocks < int64_t(dev->sm_count) * 16 ? blocks
                                                                       : int64_t(dev->sm_count) * 16);
    pcn::gather_points_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        xyz, int(N), idx, Q * K, total, out, dev->status_word);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PC_OK : cuda_err(e, "gather_points: launch");
}
