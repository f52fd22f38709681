// pc_filter.cuh -- the conservative candidate filter of the brute-force kNN
// and Ball Query kernels.
//
// The selection rules compare the exactly rounded squared distance
// s32 = ((dx*dx + dy*dy) + dz*dz) (8 separately rounded operations per
// pair) with a threshold tau (kNN: the current k-th s32, accepted if
// s32 <= tau; Ball Query: R2, accepted if s32 < R2).  The hot loops do not
// evaluate s32.  They evaluate, per (query q, reference x) pair,
//     t' = fma(az, z', fma(ay, y', fma(ax, x', w')))        3 FMAs
// with coordinates centred on a point c of the cloud, x' = fl(x - c),
// q' = fl(q - c), a = -2 q' (exact), w' = fl(|x'|^2 (1 - 2^-17)) per
// reference, and let a pair through when t' <= thr, where
//     thr = fl(fl(tau (1 + 2^-20)) - fl(qq (1 - 2^-19))) + 2^-120,
//     qq = |q'|^2 (float FMA chain).
// Every pair that passes is re-evaluated with the exact s32 from the raw
// coordinates, so the filter only decides which pairs are looked at.
//
// Why no pair with s32 <= tau is rejected (u = 2^-24; W = |x'|^2, QQ = |q'|^2
// exactly):
//  * s32 >= D^2 (1 - 5u) - 5 * 2^-150 for D = |x - q| (each rounding is
//    relative, or absolute below 2^-126; a difference that underflows is
//    exact), so s32 <= tau gives D^2 <= (tau + 5 * 2^-150) / (1 - 5u).
//  * Centring moves each coordinate by at most u |.|, so
//    D'^2 = |x' - q'|^2 <= D^2 (1 + u) + 2.001 u (W + QQ).
//  * The computed w' lies in W (1 -+ 4.01u)(1 - 2^-17); the three FMAs add
//    at most 6u (W + QQ) (every partial sum is at most (|x'| + |q'|)^2), and
//    t = W - 2 q'.x' = D'^2 - QQ, so with 2^-17 = 128u > 12.02u
//        t' <= D^2 (1 + u) - QQ (1 - 8.01u) <= tau (1 + 6.1u) + 6 * 2^-150
//              - qq (1 - 11.02u)            (qq >= QQ (1 - 3u)).
//  * The float evaluation of thr is at least tau (1 + 13.9u)
//    - qq (1 - 29.9u) before the 2^-120 term, which covers the absolute
//    terms; so t' <= thr whenever s32 <= tau.
//  * Overflow and NaN: a reference with w > 1e30 gets x' = y' = z' = 0 and
//    w' = -inf (t' = -inf, always passes); a query with qq > 1e30 gets a = 0
//    and thr = +inf (t' = w' <= +inf, always passes); below those bounds
//    |x'|, |q'| <= 1e15 and no product or sum overflows, so t' is never NaN
//    for finite coordinates and the ordered compare t' <= thr (or a running
//    minimum compared once) is exact.  A NaN coordinate gives a NaN exact
//    s32, which no selection rule accepts.
// The centre only affects how tight the filter is (the slack grows with
// |x'|^2 + |q'|^2): each consumer warp uses the centre of the bounding box
// of the cloud's first (up to) 256 points.
#pragma once

#include "pc_device.cuh"

namespace pcn {

// Packed fused multiply-add, one rounding per half: a * b + c.
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
    return __ffma2_rn(a, b, c);
}

// The filter of one query against a lane's 2P points (P packed pairs):
// bit r of the result is set when point r may satisfy the selection bound.
template <int P>
__device__ __forceinline__ unsigned filter_mask(const float2 (&x)[P],
                                                const float2 (&y)[P],
                                                const float2 (&z)[P],
                                                const float2 (&w)[P],
                                                float4 axy, float4 azt) {
    unsigned m = 0;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        float2 v = fma2_rn(x[p], make_float2(axy.x, axy.y), w[p]);
        v = fma2_rn(y[p], make_float2(axy.z, axy.w), v);
        v = fma2_rn(z[p], make_float2(azt.x, azt.y), v);
        m |= (v.x <= azt.z ? 1u : 0u) << (2 * p);
        m |= (v.y <= azt.z ? 1u : 0u) << (2 * p + 1);
    }
    return m;
}

// Any of the lane's 2P points passing the filter (the hot-loop form: a
// running minimum, compared once).
template <int P>
__device__ __forceinline__ bool filter_any(const float2 (&x)[P],
                                           const float2 (&y)[P],
                                           const float2 (&z)[P],
                                           const float2 (&w)[P], float4 axy,
                                           float4 azt) {
    float m = __int_as_float(0x7f800000);
#pragma unroll
    for (int p = 0; p < P; ++p) {
        float2 v = fma2_rn(x[p], make_float2(axy.x, axy.y), w[p]);
        v = fma2_rn(y[p], make_float2(axy.z, axy.w), v);
        v = fma2_rn(z[p], make_float2(azt.x, azt.y), v);
        m = fmin3(m, v.x, v.y);
    }
    return m <= azt.z;
}

__device__ __forceinline__ unsigned filter_mask8(const float2 (&x)[4],
                                                 const float2 (&y)[4],
                                                 const float2 (&z)[4],
                                                 const float2 (&w)[4],
                                                 float4 axy, float4 azt) {
    return filter_mask<4>(x, y, z, w, axy, azt);
}

__device__ __forceinline__ bool filter_any8(const float2 (&x)[4],
                                            const float2 (&y)[4],
                                            const float2 (&z)[4],
                                            const float2 (&w)[4], float4 axy,
                                            float4 azt) {
    return filter_any<4>(x, y, z, w, axy, azt);
}

struct FilterFrame {
    float cx, cy, cz;
};

// Centre of the bounding box of points [0, n) of `cloud` (n <= 256 is read;
// point i at cloud[stride * i]), computed by one full warp; (0, 0, 0) for an
// empty cloud.
__device__ __forceinline__ FilterFrame filter_frame(const float *cloud, int n,
                                                    int stride = 3) {
    const unsigned full = 0xffffffffu;
    const int lane = static_cast<int>(lane_id());
    const float inf = __int_as_float(0x7f800000);
    float lo[3] = {inf, inf, inf}, hi[3] = {-inf, -inf, -inf};
    const int m = min(n, 256);
    for (int i = lane; i < m; i += 32) {
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            const float v = cloud[size_t(i) * stride + a];
            lo[a] = fminf(lo[a], v);
            hi[a] = fmaxf(hi[a], v);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int a = 0; a < 3; ++a) {
            lo[a] = fminf(lo[a], __shfl_xor_sync(full, lo[a], o));
            hi[a] = fmaxf(hi[a], __shfl_xor_sync(full, hi[a], o));
        }
    }
    FilterFrame f{0.f, 0.f, 0.f};
    if (m > 0) {
        f.cx = __fmul_rn(__fadd_rn(lo[0], hi[0]), 0.5f);
        f.cy = __fmul_rn(__fadd_rn(lo[1], hi[1]), 0.5f);
        f.cz = __fmul_rn(__fadd_rn(lo[2], hi[2]), 0.5f);
        // a centre that overflowed (coordinates near the float range) is
        // replaced by the origin: any centre is correct, only tightness varies
        if (!(fabsf(f.cx) <= 1e38f) || !(fabsf(f.cy) <= 1e38f) ||
            !(fabsf(f.cz) <= 1e38f))
            f = FilterFrame{0.f, 0.f, 0.f};
    }
    return f;
}

// |v|^2 of a centred point by an FMA chain (any rounding order is covered).
__device__ __forceinline__ float filter_norm2(float x, float y, float z) {
    return __fmaf_rn(z, z, __fmaf_rn(y, y, __fmul_rn(x, x)));
}

// A centred reference for the filter: w' = |x'|^2 (1 - 2^-17); beyond 1e30
// the coordinates become 0 and w' = -inf (the point always passes).
__device__ __forceinline__ float filter_ref(float &xp, float &yp, float &zp) {
    const float w = filter_norm2(xp, yp, zp);
    if (w <= 1e30f) return __fmul_rn(w, 1.0f - 0x1p-17f);
    xp = yp = zp = 0.0f;
    return -__int_as_float(0x7f800000);
}

// The query side: a = -2 q' per axis (0 when |q'|^2 > 1e30, where the
// threshold is +inf) and qq = |q'|^2.
__device__ __forceinline__ float filter_query(float xp, float yp, float zp,
                                              float &ax, float &ay, float &az) {
    const float qq = filter_norm2(xp, yp, zp);
    const bool big = !(qq <= 1e30f);
    ax = big ? 0.0f : -2.0f * xp;
    ay = big ? 0.0f : -2.0f * yp;
    az = big ? 0.0f : -2.0f * zp;
    return qq;
}

// The pass threshold for a query with qq = |q'|^2 and selection bound tau.
__device__ __forceinline__ float filter_threshold(float tau, float qq) {
    const float inf = __int_as_float(0x7f800000);
    if (!(qq <= 1e30f) || !(tau <= 3e38f)) return inf;
    const float d = __fsub_rn(__fmul_rn(tau, 1.0f + 0x1p-20f),
                              __fmul_rn(qq, 1.0f - 0x1p-19f));
    return __fadd_rn(d, 0x1p-120f);
}

}  // namespace pcn
