// quat_short.cuh -- short sequences: the whole sequence of a few lanes in one
// CTA, held in registers and scanned across the CTA's threads.  No other CTA
// is waited on, nothing is kept between launches and no workspace is used:
// one read of every input, one write of every output, one launch.
//
// The scan and its backward are those of the Mamba-3 page, "Gradient math"
// section: cum[t] = q_t (x) cum[t-1] with cum[-1] = init, and the cotangent
// recurrence G[t] = d_cum[t] + conj(q_{t+1}) (x) G[t+1], d_q[t] = G[t] (x)
// conj(cum[t-1]), d_init = conj(q_0) (x) G[0].
#pragma once

#include "quat_common.cuh"
#include "quat_cumprod.h"

namespace qs {

// ---------------------------------------------------------------------------
// CTA g = (batch entry b, lane group): LT lanes, LT * NS threads.  Thread
// (l, s) = (tid % LT, tid / LT) holds lane l's steps [s * R, s * R + R) (steps
// at or past S read as the identity, with a zero cotangent, and are not
// written), so the CTA covers S <= NS * R.  A warp holds 32 / LT segments of
// LT adjacent lanes: every load and store of a step is LT * 16 contiguous
// bytes per segment.
//
// The scan across segments runs on one warp per lane (warps 0 .. LT - 1):
// thread j of lane l2's warp composes segments [j * SPT, (j + 1) * SPT),
// SPT = NS / 32, serially, the 32 compositions are scanned with five shuffle
// rounds, and the thread writes the prefix entering each of its segments back
// into the table.  The other warps wait at the block barrier.
// ---------------------------------------------------------------------------
template <int LT, int NS>
struct ShortShape {
    static constexpr int NT = LT * NS;    // threads
    static constexpr int SPT = NS / 32;   // segments a scan thread composes
    static_assert(NS % 32 == 0 && NT % 32 == 0 && NT <= 1024, "segments per lane: whole warps; at most 1024 threads");
};

__device__ __forceinline__ float4 shfl_up4(const float4 v, int d) {
    return make_float4(__shfl_up_sync(0xffffffffu, v.x, d), __shfl_up_sync(0xffffffffu, v.y, d),
                       __shfl_up_sync(0xffffffffu, v.z, d), __shfl_up_sync(0xffffffffu, v.w, d));
}
__device__ __forceinline__ float4 shfl_down4(const float4 v, int d) {
    return make_float4(__shfl_down_sync(0xffffffffu, v.x, d), __shfl_down_sync(0xffffffffu, v.y, d),
                       __shfl_down_sync(0xffffffffu, v.z, d), __shfl_down_sync(0xffffffffu, v.w, d));
}

// init of lane hj of batch entry b: an element of the I/O type at
// init[b * stride + hj], or (f32) a float4 there (the saved carries).
template <typename IO>
__device__ __forceinline__ float4 short_init(const void *init, long long stride, bool f32, int b, int hj) {
    const long long i = static_cast<long long>(b) * stride + hj;
    if (f32) return __ldg(reinterpret_cast<const float4 *>(init) + i);
    return IO::get(reinterpret_cast<const typename IO::elem *>(init)[i]);
}

// Forward.  carries (optional): [B, ceil(S / QS_CARRY_STEPS), HJ] float4, the
// cum entering every QS_CARRY_STEPS-step chunk (init for the first).
template <typename IO, int LT, int NS, int R>
__global__ void __launch_bounds__(ShortShape<LT, NS>::NT)
    quat_short_fwd_kernel(const typename IO::elem *__restrict__ q, const void *__restrict__ init,
                          long long init_stride, int init_f32, typename IO::elem *__restrict__ out,
                          float4 *__restrict__ carries, const Geometry geo) {
    using E = typename IO::elem;
    using SH = ShortShape<LT, NS>;
    static_assert(QS_CARRY_STEPS % R == 0, "a chunk of the carries is whole segments");
    __shared__ float4 tab[LT][NS + 1];
    const int tid = static_cast<int>(threadIdx.x);
    const int g = static_cast<int>(blockIdx.x), b = g / geo.NGb;
    const int hj0 = (g - b * geo.NGb) * LT;
    const long long S = geo.S;
    const int HJ = geo.HJ;

    // Walk 1: the segment's quaternions (kept in registers) and their product.
    const int l = tid % LT, s = tid / LT;
    const int hj = hj0 + l;
    const bool lane_ok = hj < HJ;
    const long long t0 = static_cast<long long>(s) * R;
    const E *src = q + (static_cast<long long>(b) * S + t0) * HJ + hj;
    float4 x[R];
#pragma unroll
    for (int k = 0; k < R; ++k)
        x[k] = (lane_ok && t0 + k < S) ? IO::get(__ldcs(src + static_cast<long long>(k) * HJ)) : q_ident();
    float4 A = x[0];
#pragma unroll
    for (int k = 1; k < R; ++k) A = q_mul(x[k], A);
    tab[l][s] = A;
    __syncthreads();

    // Scan across the segments of each lane: tab[l][s] becomes the cum just
    // before segment s.
    if (tid < LT * 32) {
        constexpr int SPT = SH::SPT;
        const int l2 = tid >> 5, j = tid & 31;
        float4 *row = &tab[l2][j * SPT];
        float4 a = row[0];   // the thread's segments, composed
#pragma unroll
        for (int i = 1; i < SPT; ++i) a = q_mul(row[i], a);
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {   // a = composition of threads 0 .. j
            const float4 y = shfl_up4(a, d);
            if (j >= d) a = q_mul(a, y);
        }
        const float4 e = shfl_up4(a, 1);
        float4 X = hj0 + l2 < HJ ? short_init<IO>(init, init_stride, init_f32 != 0, b, hj0 + l2) : q_ident();
        if (j > 0) X = q_mul(e, X);   // the cum entering the thread's first segment
#pragma unroll
        for (int i = 0; i < SPT; ++i) {
            const float4 ai = row[i];
            row[i] = X;
            X = q_mul(ai, X);
        }
    }
    __syncthreads();

    // Walk 2: cum from the cum before the segment.
    float4 X = tab[l][s];
    if (carries != nullptr && lane_ok && t0 < S && t0 % QS_CARRY_STEPS == 0) {
        const long long Cc = (S + QS_CARRY_STEPS - 1) / QS_CARRY_STEPS;
        carries[(static_cast<long long>(b) * Cc + t0 / QS_CARRY_STEPS) * HJ + hj] = X;
    }
    E *dst = out + (static_cast<long long>(b) * S + t0) * HJ + hj;
#pragma unroll
    for (int k = 0; k < R; ++k) {
        X = q_mul(x[k], X);
        if (lane_ok && t0 + k < S) __stcs(dst + static_cast<long long>(k) * HJ, IO::put(X));
    }
}

// Backward.  Each segment's cotangent map H -> V + M (x) H (H entering its
// last step from the right, to H leaving its first step to the left:
// H <- conj(q_t) (x) (d_cum[t] + H) step by step, so M = conj(A)) is scanned
// right to left across the segments, the products A left to right from init.
template <typename IO, int LT, int NS, int R>
__global__ void __launch_bounds__(ShortShape<LT, NS>::NT)
    quat_short_bwd_kernel(const typename IO::elem *__restrict__ q, const typename IO::elem *__restrict__ d_cum,
                          const void *__restrict__ init, long long init_stride, int init_f32,
                          typename IO::elem *__restrict__ d_q, typename IO::elem *__restrict__ d_init,
                          const Geometry geo) {
    using E = typename IO::elem;
    using SH = ShortShape<LT, NS>;
    __shared__ float4 tabA[LT][NS + 1], tabV[LT][NS + 1];
    const int tid = static_cast<int>(threadIdx.x);
    const int g = static_cast<int>(blockIdx.x), b = g / geo.NGb;
    const int hj0 = (g - b * geo.NGb) * LT;
    const long long S = geo.S;
    const int HJ = geo.HJ;

    // Walk 1: q and d_cum of the segment (kept), its product and its map.
    const int l = tid % LT, s = tid / LT;
    const int hj = hj0 + l;
    const bool lane_ok = hj < HJ;
    const long long t0 = static_cast<long long>(s) * R;
    const long long off = (static_cast<long long>(b) * S + t0) * HJ + hj;
    float4 x[R], gv[R];   // q; d_cum, then G
#pragma unroll
    for (int k = 0; k < R; ++k) {
        const bool in = lane_ok && t0 + k < S;
        x[k] = in ? IO::get(__ldcs(q + off + static_cast<long long>(k) * HJ)) : q_ident();
        gv[k] = in ? IO::get(__ldcs(d_cum + off + static_cast<long long>(k) * HJ)) : q_zero();
    }
    {
        float4 A = x[0];
#pragma unroll
        for (int k = 1; k < R; ++k) A = q_mul(x[k], A);
        float4 V = q_zero();
#pragma unroll
        for (int k = R - 1; k >= 0; --k) V = q_mul_cl(x[k], q_add(gv[k], V));
        tabA[l][s] = A;
        tabV[l][s] = V;
    }
    __syncthreads();

    // Scans across the segments of each lane: tabA[l][s] becomes the cum just
    // before segment s, tabV[l][s] the H entering its last step from the right.
    if (tid < LT * 32) {
        constexpr int SPT = SH::SPT;
        const int l2 = tid >> 5, j = tid & 31;
        float4 *rowA = &tabA[l2][j * SPT], *rowV = &tabV[l2][j * SPT];
        // The thread's segments composed: product a, and map (v, m) from the H
        // entering the last one to the H leaving the first (m = conj(a)).
        float4 a = rowA[0], v = rowV[0], m = q_conj(a);
#pragma unroll
        for (int i = 1; i < SPT; ++i) {
            const float4 ai = rowA[i];
            a = q_mul(ai, a);
            v = q_fma(v, m, rowV[i]);
            m = q_mul(m, q_conj(ai));
        }
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const float4 y = shfl_up4(a, d);
            if (j >= d) a = q_mul(a, y);   // threads 0 .. j
            // (v, m) = map of threads [j, j + 2d): this thread's part, then
            // the part d threads to the right.
            const float4 vr = shfl_down4(v, d), mr = shfl_down4(m, d);
            if (j + d < 32) {
                v = q_fma(v, m, vr);
                m = q_mul(m, mr);
            }
        }
        const float4 e = shfl_up4(a, 1), vn = shfl_down4(v, 1);
        const bool own = hj0 + l2 < HJ;
        float4 X = own ? short_init<IO>(init, init_stride, init_f32 != 0, b, hj0 + l2) : q_ident();
        if (j > 0) X = q_mul(e, X);             // the cum entering the thread's first segment
        float4 H = j < 31 ? vn : q_zero();      // the H entering its last segment: the maps to its right applied to nothing
#pragma unroll
        for (int i = SPT - 1; i >= 0; --i) {   // (reads each segment's product before it is replaced)
            const float4 vi = rowV[i];
            rowV[i] = H;
            H = q_fma(vi, q_conj(rowA[i]), H);
        }
#pragma unroll
        for (int i = 0; i < SPT; ++i) {
            const float4 ai = rowA[i];
            rowA[i] = X;
            X = q_mul(ai, X);
        }
        if (j == 0 && own)   // H leaving the first step to the left
            d_init[static_cast<long long>(b) * HJ + hj0 + l2] = IO::put(H);
    }
    __syncthreads();

    // Walk 2: G right to left from the H entering the segment, then d_q left
    // to right from the cum before it.
    float4 Hn = tabV[l][s];
#pragma unroll
    for (int k = R - 1; k >= 0; --k) {
        gv[k] = q_add(gv[k], Hn);
        Hn = q_mul_cl(x[k], gv[k]);
    }
    float4 X = tabA[l][s];
    E *dst = d_q + off;
#pragma unroll
    for (int k = 0; k < R; ++k) {
        if (lane_ok && t0 + k < S) __stcs(dst + static_cast<long long>(k) * HJ, IO::put(q_mul_cr(gv[k], X)));
        X = q_mul(x[k], X);
    }
}

}  // namespace qs
