// quat_tiles.cuh -- the aggregate / carry / apply kernels (every chunk an
// independent tile), the carry export for the forward with saved carries,
// and their shared-memory sizes.
#pragma once

#include "quat_common.cuh"

namespace qs {

// ---------------------------------------------------------------------------
// Aggregate kernel: one tile per CTA -> L_c (and W_c) of its LT lanes.
// Tiles are numbered chunk-major: tile = c * NG + g.
// ---------------------------------------------------------------------------
template <typename IO, bool BWD, int LT, int N>
__global__ void __launch_bounds__(NTHREADS)
    quat_agg_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap dmap,
                    float4 *__restrict__ aggL, float4 *__restrict__ aggW, const Geometry geo, const Control ctl) {
    constexpr int NSEG = NTHREADS / LT;
    constexpr int T = NSEG * N;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align128(smem_raw);
    using E = typename IO::elem;
    const E *Qt = reinterpret_cast<const E *>(smem);
    const E *Dt = Qt + T * LT;
    __shared__ __align__(8) uint64_t bar;
    __shared__ float4 s_a[NSEG][LT];
    __shared__ float4 s_w[BWD ? NSEG : 1][LT];

    const int tile = blockIdx.x;
    const int c = tile / geo.NG, g = tile - c * geo.NG;
    const int lane = threadIdx.x % LT, seg = threadIdx.x / LT;
    init_tile_bar(&bar);
    __syncthreads();
    stage_tile<IO, BWD, LT, T>(smem, &bar, &qmap, &dmap, geo, c, g, ctl, tile);
    wait_tile(&bar, ctl, tile);

    const int cell0 = seg * N * LT + lane;
    float4 loc = q_ident(), W = q_zero();
#pragma unroll
    for (int i = 0; i < N; ++i) {
        loc = q_mul(IO::get(Qt[cell0 + i * LT]), loc);
        if (BWD) W = q_add(W, q_mul_cl(loc, IO::get(Dt[cell0 + i * LT])));
    }
    s_a[seg][lane] = loc;
    if (BWD) s_w[seg][lane] = W;
    __syncthreads();
    if (seg == 0) {
        float4 L = q_ident();
#pragma unroll
        for (int k = 0; k < NSEG; ++k) L = q_mul(s_a[k][lane], L);
        const long long o = static_cast<long long>(c) * geo.NL + static_cast<long long>(g) * LT + lane;
        aggL[o] = L;
        if (BWD) {
            float4 V = q_zero();
#pragma unroll
            for (int k = NSEG - 1; k >= 0; --k) V = q_add(s_w[k][lane], q_mul_cl(s_a[k][lane], V));
            aggW[o] = V;
        }
    }
}

// ---------------------------------------------------------------------------
// Carry kernel: per padded lane, chunk aggregates -> carries.  Block = LB
// lanes x RT = 256/LB chunk ranges; thread (r, l) folds its range, the ranges
// are combined through shared memory, then each thread writes the carries of
// its range.  carF[c] = cum[t0-1]; carH[c] = H entering chunk c from the
// right (H_{c+1}); d_init = H_0.
// ---------------------------------------------------------------------------
template <typename IO, bool BWD, int LB>
__global__ void __launch_bounds__(NTHREADS)
    quat_carry_kernel(const float4 *__restrict__ aggL, const float4 *__restrict__ aggW,
                      const typename IO::elem *__restrict__ init, float4 *__restrict__ carF,
                      float4 *__restrict__ carH, typename IO::elem *__restrict__ d_init, const Geometry geo, int LT) {
    constexpr int RT = NTHREADS / LB;
    constexpr int U = 8;   // aggregates loaded per batch (independent loads)
    __shared__ float4 xa[RT][LB];
    __shared__ float4 xm[BWD ? RT : 1][LB];
    __shared__ float4 xv[BWD ? RT : 1][LB];
    const int l = threadIdx.x % LB, r = threadIdx.x / LB;
    const int gl = blockIdx.x * LB + l;   // padded lane
    const bool in_range = gl < geo.NL;
    const int g = gl / LT, lig = gl - g * LT;
    const int b = g / geo.NGb, hj = (g - b * geo.NGb) * LT + lig;
    const bool lane_ok = in_range && hj < geo.HJ;
    const int C = geo.C;
    const long long NL = geo.NL;
    const int R = (C + RT - 1) / RT;
    const int c_lo = min(C, r * R), c_hi = min(C, c_lo + R);
    auto at = [&](int c) { return static_cast<long long>(c) * NL + gl; };

    float4 P = q_ident(), M = q_ident(), V = q_zero();
    if (in_range) {
        for (int c0 = c_lo; c0 < c_hi; c0 += U) {
            float4 Lb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) Lb[u] = (c0 + u < c_hi) ? __ldg(aggL + at(c0 + u)) : q_ident();
#pragma unroll
            for (int u = 0; u < U; ++u) P = q_mul(Lb[u], P);
        }
        if (BWD) {
            for (int c1 = c_hi; c1 > c_lo; c1 -= U) {
                float4 Lb[U], Wb[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int cc = c1 - 1 - u;
                    const bool in = cc >= c_lo;
                    Lb[u] = in ? __ldg(aggL + at(cc)) : q_ident();
                    Wb[u] = in ? __ldg(aggW + at(cc)) : q_zero();
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    V = q_add(Wb[u], q_mul_cl(Lb[u], V));
                    M = q_mul_cl(Lb[u], M);
                }
            }
        }
    }
    xa[r][l] = P;
    if (BWD) {
        xm[r][l] = M;
        xv[r][l] = V;
    }
    __syncthreads();
    if (!in_range) return;
    float4 carry = lane_ok ? IO::get(init[static_cast<long long>(b) * geo.HJ + hj]) : q_ident();
    for (int k = 0; k < r; ++k) carry = q_mul(xa[k][l], carry);
    float4 h = q_zero();
    if (BWD) {
        for (int k = RT - 1; k > r; --k) h = q_add(xv[k][l], q_mul(xm[k][l], h));
        if (r == 0 && lane_ok) d_init[static_cast<long long>(b) * geo.HJ + hj] = IO::put(q_add(V, q_mul(M, h)));
    }
    for (int c0 = c_lo; c0 < c_hi; c0 += U) {
        float4 Lb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) Lb[u] = (c0 + u < c_hi) ? __ldg(aggL + at(c0 + u)) : q_ident();
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (c0 + u < c_hi) carF[at(c0 + u)] = carry;
            carry = q_mul(Lb[u], carry);
        }
    }
    if (BWD) {
        for (int c1 = c_hi; c1 > c_lo; c1 -= U) {
            float4 Lb[U], Wb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = c1 - 1 - u;
                const bool in = cc >= c_lo;
                Lb[u] = in ? __ldg(aggL + at(cc)) : q_ident();
                Wb[u] = in ? __ldg(aggW + at(cc)) : q_zero();
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = c1 - 1 - u;
                if (cc >= c_lo) carH[at(cc)] = h;
                h = q_add(Wb[u], q_mul_cl(Lb[u], h));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Carry kernel for many chunks per lane: a block takes LPB adjacent padded
// lanes, and thread (r, l) folds chunk range r (about C / (256 / LPB) chunks)
// of lane l; the 256 / LPB range products (and affine range maps) of a lane
// are combined by a log-depth scan in shared memory, then every thread writes
// the carries of its range.  Same outputs as quat_carry_kernel.  The
// aggregates are stored [chunk][lane], so adjacent lanes share the 32-byte
// sectors a warp's loads touch.
// ---------------------------------------------------------------------------
template <typename IO, bool BWD, int LPB>
__global__ void __launch_bounds__(NTHREADS)
    quat_carry_scan_kernel(const float4 *__restrict__ aggL, const float4 *__restrict__ aggW,
                           const typename IO::elem *__restrict__ init, float4 *__restrict__ carF,
                           float4 *__restrict__ carH, typename IO::elem *__restrict__ d_init, const Geometry geo,
                           int LT) {
    constexpr int U = 8;                // aggregates loaded per batch (independent loads)
    constexpr int RT = NTHREADS / LPB;  // chunk ranges per lane
    __shared__ float4 sP[RT][LPB];
    __shared__ float4 sM[BWD ? RT : 1][LPB];
    __shared__ float4 sV[BWD ? RT : 1][LPB];
    const int l = static_cast<int>(threadIdx.x) % LPB, r = static_cast<int>(threadIdx.x) / LPB;
    const int gl = static_cast<int>(blockIdx.x) * LPB + l;   // padded lane
    const bool in_range = gl < geo.NL;
    const int g = gl / LT, lig = gl - g * LT;
    const int b = g / geo.NGb, hj = (g - b * geo.NGb) * LT + lig;
    const bool lane_ok = in_range && hj < geo.HJ;
    const int C = geo.C;
    const long long NL = geo.NL;
    const int R = (C + RT - 1) / RT;
    const int c_lo = in_range ? min(C, r * R) : 0, c_hi = in_range ? min(C, c_lo + R) : 0;
    auto at = [&](int c) { return static_cast<long long>(c) * NL + gl; };

    // This range as a product P and (backward) as the map h -> V + M (x) h.
    float4 P = q_ident(), M = q_ident(), V = q_zero();
    for (int c0 = c_lo; c0 < c_hi; c0 += U) {
        float4 Lb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) Lb[u] = (c0 + u < c_hi) ? __ldg(aggL + at(c0 + u)) : q_ident();
#pragma unroll
        for (int u = 0; u < U; ++u) P = q_mul(Lb[u], P);
    }
    if (BWD) {
        for (int c1 = c_hi; c1 > c_lo; c1 -= U) {
            float4 Lb[U], Wb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = c1 - 1 - u;
                const bool in = cc >= c_lo;
                Lb[u] = in ? __ldg(aggL + at(cc)) : q_ident();
                Wb[u] = in ? __ldg(aggW + at(cc)) : q_zero();
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                V = q_add(Wb[u], q_mul_cl(Lb[u], V));
                M = q_mul_cl(Lb[u], M);
            }
        }
    }
    // Inclusive scans over the ranges of a lane: products of ranges 0..r
    // (later on the left) and maps of ranges r..RT-1 (range r applied last).
    sP[r][l] = P;
    if (BWD) {
        sM[r][l] = M;
        sV[r][l] = V;
    }
    __syncthreads();
    for (int d = 1; d < RT; d <<= 1) {
        const float4 oP = r >= d ? sP[r - d][l] : q_ident();
        float4 oM = q_ident(), oV = q_zero();
        if (BWD && r + d < RT) {
            oM = sM[r + d][l];
            oV = sV[r + d][l];
        }
        __syncthreads();
        if (r >= d) {
            P = q_mul(P, oP);
            sP[r][l] = P;
        }
        if (BWD && r + d < RT) {
            V = q_add(V, q_mul(M, oV));
            M = q_mul(M, oM);
            sM[r][l] = M;
            sV[r][l] = V;
        }
        __syncthreads();
    }
    if (!in_range) return;   // (after the last barrier)
    const float4 init4 = lane_ok ? IO::get(init[static_cast<long long>(b) * geo.HJ + hj]) : q_ident();
    float4 carry = r > 0 ? q_mul(sP[r - 1][l], init4) : init4;   // cum just before range r
    float4 h = q_zero();                                          // H entering range r from the right
    if (BWD) {
        if (r + 1 < RT) h = sV[r + 1][l];
        if (r == 0 && lane_ok) d_init[static_cast<long long>(b) * geo.HJ + hj] = IO::put(sV[0][l]);
    }
    for (int c0 = c_lo; c0 < c_hi; c0 += U) {
        float4 Lb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) Lb[u] = (c0 + u < c_hi) ? __ldg(aggL + at(c0 + u)) : q_ident();
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (c0 + u < c_hi) carF[at(c0 + u)] = carry;
            carry = q_mul(Lb[u], carry);
        }
    }
    if (BWD) {
        for (int c1 = c_hi; c1 > c_lo; c1 -= U) {
            float4 Lb[U], Wb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = c1 - 1 - u;
                const bool in = cc >= c_lo;
                Lb[u] = in ? __ldg(aggL + at(cc)) : q_ident();
                Wb[u] = in ? __ldg(aggW + at(cc)) : q_zero();
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = c1 - 1 - u;
                if (cc >= c_lo) carH[at(cc)] = h;
                h = q_add(Wb[u], q_mul_cl(Lb[u], h));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Apply kernel: one tile per CTA, in reverse tile order.  Forward:
// cum[t] = local_t (x) F_c.  Backward: reverse pass G = d_cum + H,
// d_q = G (x) conj(cum[t-1]), H = conj(q_t) (x) G.
// ---------------------------------------------------------------------------
template <typename IO, bool BWD, int LT, int N>
__global__ void __launch_bounds__(NTHREADS)
    quat_apply_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap dmap,
                      const float4 *__restrict__ carF, const float4 *__restrict__ carH,
                      typename IO::elem *__restrict__ out,
                      const Geometry geo, const Control ctl) {
    constexpr int NSEG = NTHREADS / LT;
    constexpr int T = NSEG * N;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align128(smem_raw);
    using E = typename IO::elem;
    const E *Qt = reinterpret_cast<const E *>(smem);
    const E *Dt = Qt + T * LT;
    __shared__ __align__(8) uint64_t bar;
    __shared__ float4 s_a[NSEG][LT];
    __shared__ float4 s_w[BWD ? NSEG : 1][LT];
    __shared__ float4 s_cf[LT];
    __shared__ float4 s_ch[BWD ? LT : 1];

    const int tile = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);   // reverse order
    const int c = tile / geo.NG, g = tile - c * geo.NG;
    const int lane = threadIdx.x % LT, seg = threadIdx.x / LT;
    init_tile_bar(&bar);
    __syncthreads();
    stage_tile<IO, BWD, LT, T>(smem, &bar, &qmap, &dmap, geo, c, g, ctl, -1);
    const long long o = static_cast<long long>(c) * geo.NL + static_cast<long long>(g) * LT + lane;
    if (seg == 0) {   // carries of this chunk (their loads overlap the tile load)
        s_cf[lane] = __ldg(carF + o);
        if (BWD) s_ch[lane] = __ldg(carH + o);
    }
    wait_tile(&bar, ctl, tile);

    const int b = g / geo.NGb, hj = (g - b * geo.NGb) * LT + lane;
    const bool lane_ok = hj < geo.HJ;
    const long long t0 = static_cast<long long>(c) * T + seg * N;
    const int cell0 = seg * N * LT + lane;
    E *dst = out + (static_cast<long long>(b) * geo.S + t0) * geo.HJ + hj;
    if (!BWD) {
        float4 x[N];
        float4 loc = q_ident();
#pragma unroll
        for (int i = 0; i < N; ++i) {
            loc = q_mul(IO::get(Qt[cell0 + i * LT]), loc);
            x[i] = loc;
        }
        s_a[seg][lane] = loc;
        __syncthreads();
        float4 X = s_cf[lane];   // cum just before this segment
        for (int k = 0; k < seg; ++k) X = q_mul(s_a[k][lane], X);
        if (lane_ok) {
#pragma unroll
            for (int i = 0; i < N; ++i)
                if (t0 + i < geo.S) __stcs(dst + static_cast<long long>(i) * geo.HJ, IO::put(q_mul(x[i], X)));
        }
    } else {
        float4 lp[N];
        float4 loc = q_ident(), W = q_zero();
#pragma unroll
        for (int i = 0; i < N; ++i) {
            lp[i] = loc;
            loc = q_mul(IO::get(Qt[cell0 + i * LT]), loc);
            W = q_add(W, q_mul_cl(loc, IO::get(Dt[cell0 + i * LT])));
        }
        s_a[seg][lane] = loc;
        s_w[seg][lane] = W;
        __syncthreads();
        float4 X = s_cf[lane];
        for (int k = 0; k < seg; ++k) X = q_mul(s_a[k][lane], X);
        float4 Hn = s_ch[lane];
        for (int k = NSEG - 1; k > seg; --k) Hn = q_add(s_w[k][lane], q_mul_cl(s_a[k][lane], Hn));
#pragma unroll
        for (int i = N - 1; i >= 0; --i) {
            const float4 G = q_add(IO::get(Dt[cell0 + i * LT]), Hn);
            if (lane_ok && t0 + i < geo.S)
                __stcs(dst + static_cast<long long>(i) * geo.HJ, IO::put(q_mul_cr(G, q_mul(lp[i], X))));
            Hn = q_mul_cl(IO::get(Qt[cell0 + i * LT]), G);
        }
    }
}


// Copies the chunk carries the carry kernel left in the workspace
// (chunk-major, padded lanes) to the caller's [B, C, H*J] layout.
__global__ void __launch_bounds__(NTHREADS)
    quat_export_carries_kernel(const float4 *__restrict__ carF, float4 *__restrict__ carries, const Geometry geo,
                               int LT, long long total) {
    const long long i = static_cast<long long>(blockIdx.x) * NTHREADS + threadIdx.x;
    if (i >= total) return;
    const long long bc = i / geo.HJ;
    const int hj = static_cast<int>(i - bc * geo.HJ);
    const int b = static_cast<int>(bc / geo.C), c = static_cast<int>(bc - static_cast<long long>(b) * geo.C);
    const long long g = static_cast<long long>(b) * geo.NGb + hj / LT;
    carries[i] = carF[static_cast<long long>(c) * geo.NL + g * LT + hj % LT];
}


// Shared memory of a tile kernel (dynamic part).
__host__ __device__ constexpr size_t tile_smem_bytes(bool bwd, int lt, int n, int eb = 16) {
    return 128 + size_t(bwd ? 2 : 1) * (NTHREADS / lt) * n * lt * eb;
}

}  // namespace qs
