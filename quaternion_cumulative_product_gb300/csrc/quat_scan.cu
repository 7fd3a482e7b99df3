// quat_scan.cu -- GB300 (sm_103a) kernels and C ABI of the quaternion
// cumulative-product scan and its recompute-based backward.
//
// The operation follows burn-mamba `mamba3/quat_scan/backward.rs`, module
// documentation "Gradient math": cum[t] = q_t (x) cum[t-1] (cum[-1] = init),
// the per-factor VJP rule, the reverse recurrence
// G[t] = d_cum[t] + conj(q_{t+1}) (x) G[t+1] and its closed form with the
// prefix product P_t and the suffix sum S[t] = sum_{s>=t} conj(P_s) (x) d_cum[s].
//
// Design (one GPU, HBM-bound; no tensor cores -- there is no dense contraction):
//
//  * Chunk = T consecutive steps of one lane group (LT lanes of one batch
//    entry, 16*LT contiguous bytes per step), staged into shared memory by
//    one 3-D TMA load per operand.  Thread (seg, lane) owns N consecutive
//    steps of one lane; NSEG segments per chunk.  TMA fills the parts of a
//    chunk past the sequence end or past the last lane with zeros, and a zero
//    step is exactly the padding the scan needs.
//
//  * Chunk aggregates (the page's factorisation):
//      L_c = q_{t1-1} (x) ... (x) q_{t0}                      (chunk product)
//      W_c = sum_{s in c} conj(local_s) (x) d_cum[s]          (backward only)
//    with local_s = q_s (x) ... (x) q_{t0}.  With H[t] = conj(q_t) (x) G[t]
//    (the cotangent step t hands to cum[t-1]), a chunk maps the H entering
//    from its right end to the H at its first step by
//      H_c = W_c + conj(L_c) (x) H_{c+1},
//    which is the page's suffix-sum factorisation
//    conj(P_s) = conj(P_{c-1}) (x) conj(local_s), and composes the literal
//    reverse recurrence, so it is exact for all quaternions.  d_init = H_0.
//    The forward carry into chunk c is F_c = cum[t0-1] = L_{c-1} (x) F_{c-1},
//    F_0 = init.
//
//  * Two designs; each call picks one from the number of lane groups.
//    Walk (one kernel): one CTA per lane group streams the whole sequence
//    through a TMA ring and keeps the carries between chunks itself -- the
//    forward reads q once and writes cum once; the backward walks forward
//    over q for the carries, then backward over q and d_cum.
//    Aggregate / carry / apply (three kernels), for too few lane groups to
//    fill the GPU: every chunk is an independent tile --
//      aggregate: one tile per CTA -> L_c (and W_c);
//      carry:     per lane, chunk aggregates -> carries F_c (and H_{c+1},
//                 d_init): 32 lanes per block over 8 chunk ranges, or for
//                 many chunks one block per lane with a scan over 256 ranges;
//      apply:     one tile per CTA, tiles in reverse order (the most recently
//                 read tiles are still in L2) -> cum (or d_q).
//    None of these kernels waits on another CTA.  A third, single-pass
//    forward (chained scan with decoupled look-back across CTAs) is compiled
//    as a configuration to force; it measured slower than both designs.
//
//  * Every tensor layout is [B, S, H, J, 4]; the kernels are templated on the
//    element type in memory (four fp32, or four bfloat16), and compute in fp32.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "quat_cumprod.h"
#include "quat_device.cuh"

namespace qs {

constexpr int NTHREADS = 256;   // threads per CTA of every kernel but the walks

// Device status of one (device, stream) workspace.
struct __align__(256) WsHeader {
    unsigned int err_code;        // 1 once a wait ran out (cleared by quat_cumprod_status)
    unsigned int err_count;       // number of waits that ran out
    unsigned long long err_item;  // first tile whose wait ran out
};

struct Geometry {
    long long S;   // sequence length
    int HJ;        // lanes per batch entry (H*J)
    int NGb;       // lane groups per batch entry
    int NG;        // lane groups in total
    int C;         // chunks along the sequence
    int NL;        // padded lanes (NG * LT): aggregates of chunk c start at c * NL
};

struct Control {
    WsHeader *hdr;
    int stall_tile;                  // test hook: this tile's wait never completes
    unsigned long long timeout_ns;   // limit of every device-side wait
};

__device__ __forceinline__ unsigned char *align128(unsigned char *p) {
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 127) & ~uintptr_t(127));
}

__device__ void record_error(WsHeader *h, int item) {
    if (atomicCAS(&h->err_code, 0u, 1u) == 0u) h->err_item = static_cast<unsigned long long>(item);
    atomicAdd(&h->err_count, 1u);
}

// Waits for the tile's TMA copies.  Bounded: after ctl.timeout_ns the error is
// recorded and the CTA carries on with whatever the stage holds (its outputs
// are then invalid, and quat_cumprod_status reports QS_ERR_TIMEOUT).
__device__ __forceinline__ void wait_tile(uint64_t *bar, const Control &ctl, int tile) {
    if (mbar_try_wait(bar, 0)) return;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, 0)) {
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            if (threadIdx.x == 0) record_error(ctl.hdr, tile);
            return;
        }
    }
}

// Thread 0 initialises the tile's barrier; the barrier must be visible to the
// whole CTA (and to the TMA unit) before the copy is issued.
__device__ __forceinline__ void init_tile_bar(uint64_t *bar) {
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
}

// Thread 0 stages the tile (q, and d_cum for the backward) of lane group g,
// chunk c.  The test hook makes the barrier of tile `tile` (>= 0; the apply
// kernel passes -1) expect 16 bytes that never come.
template <typename IO, bool BWD, int LT, int T>
__device__ __forceinline__ void stage_tile(unsigned char *dst, uint64_t *bar, const CUtensorMap *qmap,
                                           const CUtensorMap *dmap, const Geometry &geo, int c, int g,
                                           const Control &ctl, int tile) {
    constexpr uint32_t BYTES = T * LT * IO::bytes;
    if (threadIdx.x == 0) {
        const int b = g / geo.NGb, x = (g - b * geo.NGb) * LT * 4;
        const uint32_t extra = (tile >= 0 && tile == ctl.stall_tile) ? 16u : 0u;
        mbar_arrive_expect_tx(bar, (BWD ? 2 : 1) * BYTES + extra);
        tma_load_3d(dst, qmap, x, c * T, b, bar);
        if (BWD) tma_load_3d(dst + BYTES, dmap, x, c * T, b, bar);
    }
}

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
// Carry kernel for many chunks per lane: one block per padded lane, thread r
// folds the chunk range r (about C / 256 chunks); the 256 range products (and
// affine range maps) are combined by a log-depth scan in shared memory, then
// every thread writes the carries of its range.  Same outputs as
// quat_carry_kernel.
// ---------------------------------------------------------------------------
template <typename IO, bool BWD>
__global__ void __launch_bounds__(NTHREADS)
    quat_carry_scan_kernel(const float4 *__restrict__ aggL, const float4 *__restrict__ aggW,
                           const typename IO::elem *__restrict__ init, float4 *__restrict__ carF,
                           float4 *__restrict__ carH, typename IO::elem *__restrict__ d_init, const Geometry geo,
                           int LT) {
    constexpr int U = 8;   // aggregates loaded per batch (independent loads)
    __shared__ float4 sP[NTHREADS];
    __shared__ float4 sM[BWD ? NTHREADS : 1];
    __shared__ float4 sV[BWD ? NTHREADS : 1];
    const int gl = static_cast<int>(blockIdx.x);   // padded lane
    const int r = threadIdx.x;
    const int g = gl / LT, lig = gl - g * LT;
    const int b = g / geo.NGb, hj = (g - b * geo.NGb) * LT + lig;
    const bool lane_ok = hj < geo.HJ;
    const int C = geo.C;
    const long long NL = geo.NL;
    const int R = (C + NTHREADS - 1) / NTHREADS;
    const int c_lo = min(C, r * R), c_hi = min(C, c_lo + R);
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
    // Inclusive scans over the ranges: products of ranges 0..r (later on the
    // left) and maps of ranges r..255 (range r applied last).
    sP[r] = P;
    if (BWD) {
        sM[r] = M;
        sV[r] = V;
    }
    __syncthreads();
    for (int d = 1; d < NTHREADS; d <<= 1) {
        const float4 oP = r >= d ? sP[r - d] : q_ident();
        float4 oM = q_ident(), oV = q_zero();
        if (BWD && r + d < NTHREADS) {
            oM = sM[r + d];
            oV = sV[r + d];
        }
        __syncthreads();
        if (r >= d) {
            P = q_mul(P, oP);
            sP[r] = P;
        }
        if (BWD && r + d < NTHREADS) {
            V = q_add(V, q_mul(M, oV));
            M = q_mul(M, oM);
            sM[r] = M;
            sV[r] = V;
        }
        __syncthreads();
    }
    const float4 init4 = lane_ok ? IO::get(init[static_cast<long long>(b) * geo.HJ + hj]) : q_ident();
    float4 carry = r > 0 ? q_mul(sP[r - 1], init4) : init4;   // cum just before range r
    float4 h = q_zero();                                       // H entering range r from the right
    if (BWD) {
        if (r + 1 < NTHREADS) h = sV[r + 1];
        if (r == 0 && lane_ok) d_init[static_cast<long long>(b) * geo.HJ + hj] = IO::put(sV[0]);
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

// ---------------------------------------------------------------------------
// Chained-scan forward (single pass, one tile per CTA).  Tiles are numbered
// chunk-major (tile = c * NG + g) and CTAs start in that order, so a tile
// waits only on tiles that started before it.  Per lane, a tile publishes its
// chunk product L_c and, once known, its inclusive value cum at its last step
// (`incl`), each followed by that lane's status word, written with release
// semantics by the thread that wrote the value; readers acquire the status
// word before reading the value.  A tile's carry is the product of the
// aggregates of the chunks before it, back to the nearest published
// inclusive value (decoupled look-back); the NSEG segment threads of a lane
// read NSEG predecessors per round.  Status words carry the launch's epoch,
// so nothing has to be cleared between launches.  Every wait is bounded; a
// tile whose wait ran out still publishes (NaN), so no successor waits out
// its own limit because of it.
// ---------------------------------------------------------------------------
constexpr uint32_t CH_AGG = 1, CH_INCL = 2;   // status word: (epoch << 2) | state

template <typename IO, int LT, int N>
__global__ void __launch_bounds__(NTHREADS)
    quat_chain_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const typename IO::elem *__restrict__ init,
                          typename IO::elem *__restrict__ out, uint32_t *__restrict__ flags,
                          float4 *__restrict__ agg, float4 *__restrict__ incl, const Geometry geo,
                          const Control ctl, uint32_t epoch) {
    constexpr int NSEG = NTHREADS / LT;
    constexpr int T = NSEG * N;
    using E = typename IO::elem;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align128(smem_raw);
    const E *Qt = reinterpret_cast<const E *>(smem);
    __shared__ __align__(8) uint64_t bar;
    __shared__ float4 s_a[NSEG][LT];
    __shared__ float4 s_lb[NSEG][LT];       // one look-back round: a predecessor per segment
    __shared__ uint32_t s_st[NSEG][LT];
    __shared__ float4 s_x[LT];              // carry into the tile

    const int tile = static_cast<int>(blockIdx.x);
    const int c = tile / geo.NG, g = tile - c * geo.NG;
    const int lane = threadIdx.x % LT, seg = threadIdx.x / LT;
    const int b = g / geo.NGb, hj = (g - b * geo.NGb) * LT + lane;
    const bool lane_ok = hj < geo.HJ;
    init_tile_bar(&bar);
    __syncthreads();
    stage_tile<IO, false, LT, T>(smem, &bar, &qmap, &qmap, geo, c, g, ctl, tile);
    float4 init4 = q_ident();
    if (c == 0 && seg == 0 && lane_ok) init4 = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
    wait_tile(&bar, ctl, tile);

    const int cell0 = seg * N * LT + lane;
    float4 x[N];
    float4 loc = q_ident();
#pragma unroll
    for (int k = 0; k < N; ++k) {
        loc = q_mul(IO::get(Qt[cell0 + k * LT]), loc);
        x[k] = loc;
    }
    s_a[seg][lane] = loc;
    __syncthreads();
    const uint32_t tag = epoch << 2;
    const long long me = static_cast<long long>(tile) * LT + lane;
    float4 L = q_ident();
    if (seg == 0) {
#pragma unroll
        for (int k = 0; k < NSEG; ++k) L = q_mul(s_a[k][lane], L);
        if (c > 0) {   // the aggregate first: successors can use it before the carry is known
            __stcg(agg + me, L);
            st_release_u32(flags + me, tag | CH_AGG);
        }
    }
    // Look-back: acc = L_{c-1} (x) L_{c-2} (x) ... (x) incl_p.  Per round the
    // NSEG segment threads of a lane read NSEG * LB consecutive predecessors,
    // LB each (segment k: chunks base - k*LB .. base - k*LB - LB + 1), fold
    // them locally up to the first inclusive value, and segment 0 combines the
    // NSEG partial products in order.
    constexpr int LB = 4;
    float4 acc = init4;   // chunk 0: the carry is init
    bool done = c == 0;
    if (c > 0) {
        acc = q_ident();
        for (int base = c - 1;; base -= NSEG * LB) {
            float4 part = q_ident();
            uint32_t pst = 0;   // CH_INCL once the fold reached an inclusive value
#pragma unroll 1
            for (int j = 0; j < LB && pst != CH_INCL; ++j) {
                const int p = base - seg * LB - j;
                if (p < 0) break;   // chunk 0 publishes an inclusive value, so this is never needed
                const long long idx = (static_cast<long long>(p) * geo.NG + g) * LT + lane;
                uint32_t f = ld_acquire_u32(flags + idx);
                bool lost = false;
                if ((f & ~3u) != tag) {
                    const unsigned long long t0 = global_timer_ns();
                    do {
                        if (global_timer_ns() - t0 > ctl.timeout_ns) {
                            record_error(ctl.hdr, tile);
                            lost = true;
                            break;
                        }
                        f = ld_acquire_u32(flags + idx);
                    } while ((f & ~3u) != tag);
                }
                if (lost) {
                    part = q_nan();
                    pst = CH_INCL;
                } else if ((f & 3u) == CH_INCL) {
                    part = q_mul(part, __ldcg(incl + idx));
                    pst = CH_INCL;
                } else {
                    part = q_mul(part, __ldcg(agg + idx));
                }
            }
            s_lb[seg][lane] = part;
            s_st[seg][lane] = pst;
            __syncthreads();
            if (seg == 0 && !done) {
#pragma unroll 1
                for (int k = 0; k < NSEG; ++k) {
                    acc = q_mul(acc, s_lb[k][lane]);
                    if (s_st[k][lane] == CH_INCL) {
                        done = true;
                        break;
                    }
                }
            }
            if (!__syncthreads_or(seg == 0 && !done)) break;
        }
    }
    if (seg == 0) {
        __stcg(incl + me, q_mul(L, acc));
        st_release_u32(flags + me, tag | CH_INCL);
        s_x[lane] = acc;
    }
    __syncthreads();
    float4 X = s_x[lane];   // cum just before this segment
#pragma unroll
    for (int k = 0; k < NSEG - 1; ++k)
        if (k < seg) X = q_mul(s_a[k][lane], X);
    const long long t0 = static_cast<long long>(c) * T + seg * N;
    E *dst = out + (static_cast<long long>(b) * geo.S + t0) * geo.HJ + hj;
    if (lane_ok && t0 + N <= geo.S) {
#pragma unroll
        for (int k = 0; k < N; ++k) __stcs(dst + static_cast<long long>(k) * geo.HJ, IO::put(q_mul(x[k], X)));
    } else if (lane_ok) {
#pragma unroll
        for (int k = 0; k < N; ++k)
            if (t0 + k < geo.S) __stcs(dst + static_cast<long long>(k) * geo.HJ, IO::put(q_mul(x[k], X)));
    }
}

// ---------------------------------------------------------------------------
// Walk kernels.  One CTA walks one lane group (LT lanes of one batch entry)
// along the whole sequence, chunk by chunk: chunk c = T steps x LT lanes is
// staged by one TMA load per operand through an NST-deep ring, thread
// (seg, lane) owns N consecutive steps of one lane (NSEG segments per chunk),
// and the carry between chunks stays in the CTA.  Nothing waits on another
// CTA.  One block barrier per chunk: what a chunk needs from the one before
// it (the carry, and in the backward the right-hand cotangent) is published
// one chunk ahead in double-buffered shared slots, and the segment aggregates
// are double-buffered as well.
//
// Forward: one pass, cum[t] = local_t (x) F_c, 32 bytes per element.
// Backward: a forward walk over q that stores the carries F_c (q loaded with
// the L2 evict-last policy), then a reverse walk over q and d_cum
// (evict-first) that folds the affine chunk maps H_c = W_c + conj(L_c) (x)
// H_{c+1} and writes d_q.  The reverse walk starts with the chunks the
// forward walk read last, so as much of q as L2 holds is read from L2 the
// second time: 48 to 64 bytes of DRAM traffic per element.
// ---------------------------------------------------------------------------

// Bounded wait on one stage of a ring; false if the wait ran out (the error is
// recorded by thread 0).
__device__ __forceinline__ bool wait_stage(uint64_t *bar, uint32_t parity, const Control &ctl, int item) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            if (threadIdx.x == 0) record_error(ctl.hdr, item);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ int ld_volatile_int(const int *p) { return *reinterpret_cast<const volatile int *>(p); }

// After a wait ran out, the ring's barriers are no longer in step with the
// loads; the kernel stops issuing loads and, before it exits, gives the loads
// it did issue a bounded time to land (so that none writes into the shared
// memory of a later CTA).
template <int NS>
__device__ __forceinline__ void drain_ring(uint64_t *bars, const int *issued, const Control &ctl) {
    if (threadIdx.x != 0) return;
    for (int s = 0; s < NS; ++s) {
        if (issued[s] == 0) continue;
        const uint32_t parity = static_cast<uint32_t>(issued[s] - 1) & 1u;
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&bars[s], parity) && global_timer_ns() - t0 <= ctl.timeout_ns) {
        }
    }
}

// `carries` (optional, may be null): [B, C, H*J] float4, the state entering
// every chunk, carries[b, c] = cum[b, c*T - 1] (init for c = 0).
template <typename IO, int LT, int NSEG, int N, int NST>
__global__ void __launch_bounds__(LT *NSEG)
    quat_walk_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const typename IO::elem *__restrict__ init,
                         typename IO::elem *__restrict__ out, float4 *__restrict__ carries, const Geometry geo,
                         const Control ctl) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr uint32_t BYTES = T * LT * IO::bytes;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    __shared__ __align__(8) uint64_t full[NST];
    __shared__ int issued[NST];   // loads issued per stage (thread 0)
    __shared__ int s_broken;
    __shared__ float4 s_a[2][NSEG][LT];   // segment products of chunk i (slot i & 1)
    __shared__ float4 s_x[2][LT];         // carry into chunk i (slot i & 1)

    const int g = static_cast<int>(blockIdx.x);
    const int b = g / geo.NGb, x0 = (g - b * geo.NGb) * LT * 4;
    const int lane = threadIdx.x % LT, seg = threadIdx.x / LT;
    const int hj = (g - b * geo.NGb) * LT + lane;
    const bool lane_ok = hj < geo.HJ;
    const int C = geo.C;

    float4 R = q_ident();   // carry into the next chunk (segment-0 threads)
    if (seg == 0 && lane_ok) R = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
    if (seg == 0) s_x[0][lane] = R;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            issued[s] = 0;
        }
        fence_mbar_init();
        s_broken = 0;
    }
    __syncthreads();
    auto issue = [&](int c) {   // thread 0: chunk c into stage c % NST
        const int st = c % NST;
        ++issued[st];
        mbar_arrive_expect_tx(&full[st], BYTES + (c * geo.NG + g == ctl.stall_tile ? 16u : 0u));
        tma_load_3d(ring + st * BYTES, &qmap, x0, c * T, b, &full[st]);
    };
    if (threadIdx.x == 0)
        for (int c = 0; c < NST && c < C; ++c) issue(c);

    const long long row0 = static_cast<long long>(b) * geo.S;
    for (int c = 0; c < C; ++c) {
        const int st = c % NST, sl = c & 1;
        const E *Qt = reinterpret_cast<const E *>(ring + st * BYTES);
        if (!ld_volatile_int(&s_broken) && !wait_stage(&full[st], (c / NST) & 1, ctl, c * geo.NG + g))
            s_broken = 1;
        float4 x[N];
        float4 loc = q_ident();
#pragma unroll
        for (int k = 0; k < N; ++k) {
            loc = q_mul(IO::get(Qt[(seg * N + k) * LT + lane]), loc);
            x[k] = loc;
        }
        s_a[sl][seg][lane] = loc;
        __syncthreads();
        if (threadIdx.x == 0 && !s_broken && c + NST < C) issue(c + NST);
        float4 P = q_ident();   // product of the earlier segments of the chunk
#pragma unroll
        for (int k = 0; k < NSEG - 1; ++k)
            if (k < seg) P = q_mul(s_a[sl][k][lane], P);
        const float4 Y = q_mul(P, s_x[sl][lane]);
        if (seg == 0) {
            if (carries != nullptr && lane_ok)
                carries[(static_cast<long long>(b) * C + c) * geo.HJ + hj] = R;   // state entering chunk c
            float4 L = q_ident();
#pragma unroll
            for (int k = 0; k < NSEG; ++k) L = q_mul(s_a[sl][k][lane], L);
            R = q_mul(L, R);
            s_x[sl ^ 1][lane] = R;
        }
        const long long t0 = static_cast<long long>(c) * T + seg * N;
        E *dst = out + (row0 + t0) * geo.HJ + hj;
        if (lane_ok && t0 + N <= geo.S) {
#pragma unroll
            for (int k = 0; k < N; ++k) __stcs(dst + static_cast<long long>(k) * geo.HJ, IO::put(q_mul(x[k], Y)));
        } else if (lane_ok) {
#pragma unroll
            for (int k = 0; k < N; ++k)
                if (t0 + k < geo.S) __stcs(dst + static_cast<long long>(k) * geo.HJ, IO::put(q_mul(x[k], Y)));
        }
    }
    if (s_broken) drain_ring<NST>(full, issued, ctl);
}

// SELF = false: after a chunk's segment aggregates are in shared memory, the
// segment-0 thread of each lane folds them once (two chains of NSEG products)
// and a second block barrier hands each segment its carry and cotangent.
// SELF = true: every thread folds its own carry (through the earlier
// segments) and cotangent (through the later ones), about NSEG-1 products,
// and the chunk needs no second barrier; segment 0 publishes the cotangent
// entering the next chunk one chunk ahead.
//
// GIVEN = true: the chunk carries come from the caller, `given` = [B, C, H*J]
// float4 with given[b, c] = cum[b, c*T - 1] (what the forward walk writes as
// `carries`); the forward walk is skipped and `init` and `carF` are unused.
template <typename IO, int LT, int NSEG, int N, int NSTF, int NSTB, bool SELF, bool GIVEN>
__global__ void __launch_bounds__(LT *NSEG)
    quat_walk_bwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap dmap,
                         const typename IO::elem *__restrict__ init, float4 *__restrict__ carF,
                         const float4 *__restrict__ given, typename IO::elem *__restrict__ d_q,
                         typename IO::elem *__restrict__ d_init, const Geometry geo, const Control ctl) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr uint32_t BQ = T * LT * IO::bytes;   // one operand of one chunk
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    __shared__ __align__(8) uint64_t fullF[NSTF];
    __shared__ __align__(8) uint64_t fullB[NSTB];
    __shared__ int issuedF[NSTF], issuedB[NSTB];
    __shared__ int s_broken;
    __shared__ float4 s_a[2][NSEG][LT];             // segment products (slot: chunk parity)
    __shared__ float4 s_w[SELF ? 2 : 1][NSEG][LT];  // segment weighted sums (reverse walk)
    __shared__ float4 s_x[SELF ? 1 : NSEG][LT];     // cum just before each segment
    __shared__ float4 s_h[SELF ? 2 : NSEG][LT];     // H entering each segment / the next chunk

    const int g = static_cast<int>(blockIdx.x);
    const int b = g / geo.NGb, x0 = (g - b * geo.NGb) * LT * 4;
    const int lane = threadIdx.x % LT, seg = threadIdx.x / LT;
    const int hj = (g - b * geo.NGb) * LT + lane;
    const bool lane_ok = hj < geo.HJ;
    const int C = geo.C;
    const long long NL = geo.NL;
    const long long col = static_cast<long long>(g) * LT + lane;   // padded lane of this thread

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTF; ++s) {
            mbar_init(&fullF[s], 1);
            issuedF[s] = 0;
        }
        for (int s = 0; s < NSTB; ++s) {
            mbar_init(&fullB[s], 1);
            issuedB[s] = 0;
        }
        fence_mbar_init();
        s_broken = 0;
    }
    __syncthreads();
    const uint64_t drop = l2_policy_evict_first();

    if constexpr (!GIVEN) {
        // ---- forward walk over q: carries F_c --------------------------------
        const uint64_t keep = l2_policy_evict_last();
        auto issueF = [&](int c) {
            const int st = c % NSTF;
            ++issuedF[st];
            mbar_arrive_expect_tx(&fullF[st], BQ + (c * geo.NG + g == ctl.stall_tile ? 16u : 0u));
            tma_load_3d_hint(ring + st * BQ, &qmap, x0, c * T, b, &fullF[st], keep);
        };
        if (threadIdx.x == 0)
            for (int c = 0; c < NSTF && c < C; ++c) issueF(c);

        float4 R = q_ident();
        if (seg == 0 && lane_ok) R = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
        for (int c = 0; c < C; ++c) {
            const int st = c % NSTF, sl = c & 1;
            const E *Qt = reinterpret_cast<const E *>(ring + st * BQ);
            if (!ld_volatile_int(&s_broken) && !wait_stage(&fullF[st], (c / NSTF) & 1, ctl, c * geo.NG + g))
                s_broken = 1;
            float4 loc = q_ident();
#pragma unroll
            for (int k = 0; k < N; ++k) loc = q_mul(IO::get(Qt[(seg * N + k) * LT + lane]), loc);
            s_a[sl][seg][lane] = loc;
            __syncthreads();
            if (threadIdx.x == 0 && !s_broken && c + NSTF < C) issueF(c + NSTF);
            if (seg == 0) {   // segment 0 carries the lane through the chunk
                carF[static_cast<long long>(c) * NL + col] = R;
#pragma unroll
                for (int k = 0; k < NSEG; ++k) R = q_mul(s_a[sl][k][lane], R);
            }
        }
    }
    __syncthreads();   // every read of the forward ring is done before the reverse ring reuses it

    // ---- reverse walk over q and d_cum: d_q, d_init --------------------------
    auto issueB = [&](int j) {   // reverse step j covers chunk C-1-j
        const int st = j % NSTB, c = C - 1 - j;
        ++issuedB[st];
        unsigned char *dst = ring + st * 2 * BQ;
        mbar_arrive_expect_tx(&fullB[st], 2 * BQ);
        tma_load_3d_hint(dst, &qmap, x0, c * T, b, &fullB[st], drop);
        tma_load_3d_hint(dst + BQ, &dmap, x0, c * T, b, &fullB[st], drop);
    };
    if (threadIdx.x == 0 && !s_broken)
        for (int j = 0; j < NSTB && j < C; ++j) issueB(j);

    float4 Hc = q_zero();   // H entering the current chunk from the right (segment-0 threads)
    // Carry into the chunk, written by this lane's segment-0 thread in the
    // forward walk; loaded one chunk ahead.
    auto carry_of = [&](int c) -> float4 {
        if constexpr (GIVEN) return lane_ok ? given[(static_cast<long long>(b) * C + c) * geo.HJ + hj] : q_ident();
        else return carF[static_cast<long long>(c) * NL + col];
    };
    float4 F_next = q_ident();
    if (SELF || seg == 0) F_next = carry_of(C - 1);
    if (SELF && seg == 0) s_h[0][lane] = Hc;
    if (SELF) __syncthreads();
    const long long row0 = static_cast<long long>(b) * geo.S;
    for (int j = 0; j < C; ++j) {
        const int c = C - 1 - j;
        const int st = j % NSTB, sl = j & 1;
        const float4 F = F_next;
        if ((SELF || seg == 0) && c > 0) F_next = carry_of(c - 1);
        const E *Qt = reinterpret_cast<const E *>(ring + st * 2 * BQ);
        const E *Dt = Qt + T * LT;
        if (!ld_volatile_int(&s_broken) && !wait_stage(&fullB[st], (j / NSTB) & 1, ctl, c * geo.NG + g))
            s_broken = 1;
        const int cell0 = seg * N * LT + lane;
        float4 qv[N], dv[N], lp[N];
        float4 loc = q_ident(), W = q_zero();
#pragma unroll
        for (int k = 0; k < N; ++k) {
            qv[k] = IO::get(Qt[cell0 + k * LT]);
            dv[k] = IO::get(Dt[cell0 + k * LT]);
            lp[k] = loc;
            loc = q_mul(qv[k], loc);
            W = q_fma_cl(W, loc, dv[k]);
        }
        const int ws = SELF ? sl : 0;
        s_a[sl][seg][lane] = loc;
        s_w[ws][seg][lane] = W;
        __syncthreads();
        if (threadIdx.x == 0 && !s_broken && j + NSTB < C) issueB(j + NSTB);
        float4 X, Hn;
        if constexpr (SELF) {
            X = F;   // through the earlier segments
#pragma unroll
            for (int k = 0; k < NSEG - 1; ++k)
                if (k < seg) X = q_mul(s_a[sl][k][lane], X);
            Hn = s_h[sl][lane];   // through the later segments
#pragma unroll
            for (int k = NSEG - 1; k > 0; --k)
                if (k > seg) Hn = q_fma_cl(s_w[ws][k][lane], s_a[sl][k][lane], Hn);
            if (seg == 0) {
                Hc = q_fma_cl(s_w[ws][0][lane], s_a[sl][0][lane], Hn);
                s_h[sl ^ 1][lane] = Hc;
                if (c == 0 && lane_ok) d_init[static_cast<long long>(b) * geo.HJ + hj] = IO::put(Hc);
            }
        } else {
            if (seg == 0) {
                // The carry forward through the segments, and H backward
                // through them: two independent chains of NSEG products.
                float4 Xs = F, h = Hc;
#pragma unroll
                for (int k = 0; k < NSEG; ++k) {
                    const int kr = NSEG - 1 - k;
                    s_x[k][lane] = Xs;
                    s_h[kr][lane] = h;
                    Xs = q_mul(s_a[sl][k][lane], Xs);
                    h = q_fma_cl(s_w[0][kr][lane], s_a[sl][kr][lane], h);
                }
                Hc = h;
                if (c == 0 && lane_ok) d_init[static_cast<long long>(b) * geo.HJ + hj] = IO::put(Hc);
            }
            __syncthreads();
            X = s_x[seg][lane];    // cum just before this segment
            Hn = s_h[seg][lane];   // H entering this segment from the right
        }
        const long long t0 = static_cast<long long>(c) * T + seg * N;
        E *dst = d_q + (row0 + t0) * geo.HJ + hj;
        if (lane_ok && t0 + N <= geo.S) {
#pragma unroll
            for (int k = N - 1; k >= 0; --k) {
                const float4 G = q_add(dv[k], Hn);
                __stcs(dst + static_cast<long long>(k) * geo.HJ, IO::put(q_mul_cr(G, q_mul(lp[k], X))));
                Hn = q_mul_cl(qv[k], G);
            }
        } else if (lane_ok) {
#pragma unroll
            for (int k = N - 1; k >= 0; --k) {
                const float4 G = q_add(dv[k], Hn);
                if (t0 + k < geo.S) __stcs(dst + static_cast<long long>(k) * geo.HJ, IO::put(q_mul_cr(G, q_mul(lp[k], X))));
                Hn = q_mul_cl(qv[k], G);
            }
        }
    }
    if (s_broken) {
        drain_ring<NSTF>(fullF, issuedF, ctl);
        drain_ring<NSTB>(fullB, issuedB, ctl);
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

// Dynamic shared memory of the walk kernels: the forward ring, or the larger
// of the backward's two rings (one operand per stage forward, two reverse).
__host__ __device__ constexpr size_t walk_fwd_smem_bytes(int lt, int nseg, int n, int nst, int eb = 16) {
    return 128 + size_t(nst) * nseg * n * lt * eb;
}
__host__ __device__ constexpr size_t walk_bwd_smem_bytes(int lt, int nseg, int n, int nstf, int nstb, int eb = 16) {
    return 128 + size_t(nstf > 2 * nstb ? nstf : 2 * nstb) * nseg * n * lt * eb;
}
}  // namespace qs

// ===========================================================================
// Host side: argument checks, workspace, tensor maps, launches, C ABI.
// ===========================================================================
namespace {

using qs::NTHREADS;

constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;

// One compiled configuration: lane-group width LT, segments per chunk NSEG
// (threads per CTA = LT * NSEG), steps per thread N.
struct Variant {
    bool walk;           // walk kernel (else aggregate / carry / apply, or chain)
    const void *agg;     // the walk kernel, or the aggregate kernel
    const void *apply;   // the apply kernel (three-kernel variants)
    bool bwd;
    int lt, nseg, n;
    size_t smem_bytes;   // dynamic shared memory per CTA
    int T() const { return nseg * n; }
    int threads() const { return lt * nseg; }
    size_t smem() const { return smem_bytes; }
    bool chain = false;  // single-pass chained scan (forward): `agg` is the kernel
};

#define QS_VARIANT(B, LT, N)                                                                        \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_agg_kernel<qs::IoF32, B, LT, N>),            \
            reinterpret_cast<const void *>(qs::quat_apply_kernel<qs::IoF32, B, LT, N>), B, LT,      \
            NTHREADS / (LT), N, qs::tile_smem_bytes(B, LT, N)                                       \
    }
#define QS_WALK_FWD(LT, NSEG, N, NST)                                                               \
    Variant {                                                                                       \
        true, reinterpret_cast<const void *>(qs::quat_walk_fwd_kernel<qs::IoF32, LT, NSEG, N, NST>), nullptr, \
            false, LT, NSEG, N, qs::walk_fwd_smem_bytes(LT, NSEG, N, NST)                           \
    }
#define QS_WALK_BWD(LT, NSEG, N, NSTF, NSTB, SELF)                                                  \
    Variant {                                                                                       \
        true, reinterpret_cast<const void *>(qs::quat_walk_bwd_kernel<qs::IoF32, LT, NSEG, N, NSTF, NSTB, SELF, false>), \
            nullptr, true, LT, NSEG, N, qs::walk_bwd_smem_bytes(LT, NSEG, N, NSTF, NSTB)            \
    }
const Variant kFwdVariants[] = {
    QS_VARIANT(false, 32, 8),          // 0: three kernels, 64-step chunks, 32 KiB tiles
    QS_VARIANT(false, 32, 4),          // 1: three kernels, 32-step chunks
    QS_VARIANT(false, 64, 8),          // 2: three kernels, 64 lanes x 32 steps
    QS_VARIANT(false, 32, 16),         // 3: three kernels, 128-step chunks
    QS_WALK_FWD(32, 8, 8, 3),          // 4: walk, 32 lanes x 64 steps, 3 x 32 KiB ring
    QS_WALK_FWD(16, 8, 8, 3),          // 5: walk, 16 lanes x 64 steps (128 threads), 3 x 16 KiB
    QS_WALK_FWD(16, 16, 8, 3),         // 6: walk, 16 lanes x 128 steps (256 threads), 3 x 32 KiB
    QS_WALK_FWD(32, 8, 4, 6),          // 7: walk, 32 lanes x 32 steps, 6 x 16 KiB
    Variant{false, reinterpret_cast<const void *>(qs::quat_chain_fwd_kernel<qs::IoF32, 32, 8>), nullptr, false,
            32, NTHREADS / 32, 8, qs::tile_smem_bytes(false, 32, 8), true},   // 8: chained scan, 64-step tiles
};
const Variant kBwdVariants[] = {
    QS_VARIANT(true, 32, 8),           // 0: three kernels, 64-step chunks, 64 KiB tiles
    QS_VARIANT(true, 32, 4),           // 1: three kernels, 32-step chunks
    QS_VARIANT(true, 64, 4),           // 2: three kernels, 64 lanes x 16 steps
    QS_VARIANT(true, 64, 8),           // 3: three kernels, 64 lanes x 32 steps
    QS_WALK_BWD(16, 8, 8, 4, 2, false),   // 4: walk, 16 lanes x 64 steps (128 threads), 64 KiB rings, one fold per lane
    QS_WALK_BWD(16, 8, 8, 6, 3, false),   // 5: walk, 16 lanes x 64 steps, 96 KiB rings
    QS_WALK_BWD(32, 8, 8, 6, 3, false),   // 6: walk, 32 lanes x 64 steps, 192 KiB rings
    QS_WALK_BWD(32, 8, 4, 6, 3, false),   // 7: walk, 32 lanes x 32 steps, 96 KiB rings
    QS_WALK_BWD(16, 8, 8, 4, 2, true),    // 8: walk, 16 lanes x 64 steps, each thread folds its own carries
    QS_WALK_BWD(32, 8, 8, 6, 3, true),    // 9: walk, 32 lanes x 64 steps, each thread folds its own carries
};
// The backward from caller-provided carries: the reverse walk alone.
const Variant kBwdGiven = Variant{true,
                                  reinterpret_cast<const void *>(qs::quat_walk_bwd_kernel<qs::IoF32, 16, 8, 8, 1, 2, false, true>),
                                  nullptr,
                                  true,
                                  16,
                                  8,
                                  8,
                                  qs::walk_bwd_smem_bytes(16, 8, 8, 1, 2)};
// bf16 I/O (fp32 arithmetic): walk kernels only.
#define QS_WALK_FWD16(LT, NSEG, N, NST)                                                             \
    Variant {                                                                                       \
        true, reinterpret_cast<const void *>(qs::quat_walk_fwd_kernel<qs::IoBF16, LT, NSEG, N, NST>), \
            nullptr, false, LT, NSEG, N, qs::walk_fwd_smem_bytes(LT, NSEG, N, NST, 8)               \
    }
#define QS_WALK_BWD16(LT, NSEG, N, NSTF, NSTB, SELF)                                                \
    Variant {                                                                                       \
        true,                                                                                       \
            reinterpret_cast<const void *>(                                                         \
                qs::quat_walk_bwd_kernel<qs::IoBF16, LT, NSEG, N, NSTF, NSTB, SELF, false>),        \
            nullptr, true, LT, NSEG, N, qs::walk_bwd_smem_bytes(LT, NSEG, N, NSTF, NSTB, 8)         \
    }
#define QS_VARIANT16(B, LT, N)                                                                      \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_agg_kernel<qs::IoBF16, B, LT, N>),           \
            reinterpret_cast<const void *>(qs::quat_apply_kernel<qs::IoBF16, B, LT, N>), B, LT,     \
            NTHREADS / (LT), N, qs::tile_smem_bytes(B, LT, N, 8)                                    \
    }
const Variant kFwdBf16Variants[] = {
    QS_WALK_FWD16(32, 8, 8, 6),            // 0: 32 lanes x 64 steps, 6 x 16 KiB ring
    QS_WALK_FWD16(16, 8, 8, 6),            // 1: 16 lanes x 64 steps (128 threads), 6 x 8 KiB
    QS_WALK_FWD16(16, 16, 8, 4),           // 2: 16 lanes x 128 steps (256 threads), 4 x 16 KiB
    QS_WALK_FWD16(32, 16, 4, 6),           // 3: 32 lanes x 64 steps (512 threads), 6 x 16 KiB
    QS_VARIANT16(false, 32, 8),            // 4: three kernels, 64-step chunks (few lane groups)
};
const Variant kBwdBf16Variants[] = {
    QS_WALK_BWD16(16, 8, 8, 8, 4, false),  // 0: 16 lanes x 64 steps (128 threads), 64 KiB rings
    QS_WALK_BWD16(16, 8, 8, 8, 4, true),   // 1: the same, each thread folds its own carries
    QS_WALK_BWD16(16, 16, 4, 8, 4, false), // 2: 16 lanes x 64 steps (256 threads), 64 KiB rings
    QS_WALK_BWD16(32, 8, 8, 8, 4, false),  // 3: 32 lanes x 64 steps (256 threads), 128 KiB rings
    QS_VARIANT16(true, 32, 8),             // 4: three kernels, 64-step chunks (few lane groups)
};
#undef QS_VARIANT16
#undef QS_WALK_FWD16
#undef QS_WALK_BWD16
constexpr int kNumFwdBf16 = sizeof(kFwdBf16Variants) / sizeof(kFwdBf16Variants[0]);
constexpr int kFwdBf16Default = 1, kBwdBf16Default = 0;   // walks; fastest measured on 8x4096x16x32
constexpr int kFwdBf16Three = 4, kBwdBf16Three = 4;       // for too few lane groups
constexpr int kNumBwdBf16 = sizeof(kBwdBf16Variants) / sizeof(kBwdBf16Variants[0]);
#undef QS_VARIANT
#undef QS_WALK_FWD
#undef QS_WALK_BWD
// Automatic choice between the two designs.  A walk keeps one CTA per lane
// group for the whole sequence, so it needs enough lane groups to keep every
// SM streaming (measured: 128 groups of 32 lanes forward and 256 groups of 16
// lanes backward already beat the three-kernel path on 152 SMs).  With fewer
// lanes -- long sequences of few lanes -- the three-kernel path, which splits
// the sequence into independent tiles, is the faster one.
constexpr int kWalkFwd = 4, kWalkBwd = 4, kThreeFwd = 0, kThreeBwd = 0;
constexpr int kNumFwd = sizeof(kFwdVariants) / sizeof(kFwdVariants[0]);
constexpr int kNumBwd = sizeof(kBwdVariants) / sizeof(kBwdVariants[0]);

std::mutex g_mu;
unsigned long long g_timeout_ns = DEFAULT_TIMEOUT_NS;
int g_stall_tile = -1;
int g_fwd_variant = -1, g_bwd_variant = -1;   // -1: automatic
int g_fwd_variant16 = -1, g_bwd_variant16 = -1;

struct DevInfo {
    int sms = 0;
    int major = 0, minor = 0;
};
std::map<int, DevInfo> g_dev;

// Library-owned scratch of one (device, stream): status block, then the
// per-call aggregate and carry arrays.
struct Workspace {
    unsigned char *base = nullptr;
    size_t bytes = 0;
    uint32_t epoch = 0;   // status words only: last epoch used
};
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;
// Status words of the chained scan, per (device, stream): an allocation of
// their own that no other kernel writes, zeroed when allocated.
std::map<std::pair<int, uintptr_t>, Workspace> g_flags;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Validates sizes; returns QS_OK, QS_ERR_DIMS, or 1 for "nothing to do".
int check_dims(int64_t B, int64_t S, int64_t H, int64_t J) {
    if (B < 0 || S < 0 || H < 0 || J < 0) return QS_ERR_DIMS;
    if (B == 0 || S == 0 || H == 0 || J == 0) return 1;
    const int64_t lim31 = (int64_t(1) << 31) - 1;
    if (B > lim31 || S > lim31 || H > lim31 || J > lim31) return QS_ERR_DIMS;
    const __int128 HJ = (__int128)H * J;
    if (HJ * 4 >= ((__int128)1 << 32) - 1) return QS_ERR_DIMS;           // TMA dimension 0
    if ((__int128)S * HJ * 16 >= ((__int128)1 << 40)) return QS_ERR_DIMS;  // TMA stride of dimension 2
    return QS_OK;
}

int device_info(DevInfo **out, int *dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &d = g_dev[dev];
    if (d.sms == 0) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            d.sms = 0;
            return QS_ERR_CUDA;
        }
        if (d.major == 10 && d.minor == 3) {
            bool ok = true;
            auto setup = [&](const Variant &v) {
                ok = ok &&
                     cudaFuncSetAttribute(v.agg, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v.smem()) ==
                         cudaSuccess;
                if (v.apply)
                    ok = ok && cudaFuncSetAttribute(v.apply, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                    (int)v.smem()) == cudaSuccess;
            };
            for (const Variant &v : kFwdVariants) setup(v);
            for (const Variant &v : kBwdVariants) setup(v);
            setup(kBwdGiven);
            for (const Variant &v : kFwdBf16Variants) setup(v);
            for (const Variant &v : kBwdBf16Variants) setup(v);
            if (!ok) {
                cudaGetLastError();
                d.sms = 0;
                return QS_ERR_CUDA;
            }
        }
    }
    if (!(d.major == 10 && d.minor == 3)) return QS_ERR_DEVICE;
    *out = &d;
    *dev_out = dev;
    return QS_OK;
}

// Returns the workspace of (device, stream) with at least `need` bytes.
int ensure_workspace(int dev, cudaStream_t stream, size_t need, unsigned char **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (w.bytes >= need) {
        *out = w.base;
        return QS_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return QS_ERR_NOMEM;
    if (w.base) {
        if (cudaStreamSynchronize(stream) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        cudaFree(w.base);
        w.base = nullptr;
        w.bytes = 0;
    }
    const size_t bytes = align_up(need + need / 4, 1 << 20);
    void *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_NOMEM;
    }
    if (cudaMemsetAsync(p, 0, sizeof(qs::WsHeader), stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p);
        return QS_ERR_CUDA;
    }
    w.base = static_cast<unsigned char *>(p);
    w.bytes = bytes;
    *out = w.base;
    return QS_OK;
}

// Status words of at least `need` bytes for a chained scan on (device,
// stream), and the epoch this launch writes into them (epoch << 2 | state).
// The words are zero when allocated; when the epochs run out they are
// cleared on the stream and the count starts again.
int chain_flags(int dev, cudaStream_t stream, size_t need, uint32_t **out, uint32_t *epoch) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_flags[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (w.bytes < need) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        if (cs != cudaStreamCaptureStatusNone) return QS_ERR_NOMEM;
        if (w.base) {
            if (cudaStreamSynchronize(stream) != cudaSuccess) {
                cudaGetLastError();
                return QS_ERR_CUDA;
            }
            cudaFree(w.base);
            w.base = nullptr;
            w.bytes = 0;
        }
        const size_t bytes = align_up(need + need / 4, 1 << 20);
        void *p = nullptr;
        if (cudaMalloc(&p, bytes) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_NOMEM;
        }
        if (cudaMemsetAsync(p, 0, bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            cudaFree(p);
            return QS_ERR_CUDA;
        }
        w.base = static_cast<unsigned char *>(p);
        w.bytes = bytes;
        w.epoch = 0;
    }
    if (w.epoch >= (1u << 30) - 1) {
        if (cudaMemsetAsync(w.base, 0, w.bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        w.epoch = 0;
    }
    *epoch = ++w.epoch;
    *out = reinterpret_cast<uint32_t *>(w.base);
    return QS_OK;
}

// 3-D view [B][S][HJ*4 floats] of a [B,S,H,J,4] tensor for TMA boxes of `lt`
// lanes x `boxh` steps.  Boxes may reach past the tensor: TMA fills those
// cells with zeros.
// `eb`: bytes of one quaternion (16 fp32, 8 bf16).
int make_map(CUtensorMap *m, const void *ptr, int64_t B, int64_t S, int64_t HJ, int lt, int boxh, int eb = 16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QS_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)(HJ * 4), (cuuint64_t)S, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)(HJ * eb), (cuuint64_t)(S * HJ * eb)};
    cuuint32_t box[3] = {(cuuint32_t)(lt * 4), (cuuint32_t)boxh, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = eb == 8 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QS_OK : QS_ERR_CUDA;
}

int pick_variant(bool bwd, int64_t B, int64_t HJ, int sms) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const int forced = bwd ? g_bwd_variant : g_fwd_variant;
        if (forced >= 0) return forced;
    }
    const Variant &w = bwd ? kBwdVariants[kWalkBwd] : kFwdVariants[kWalkFwd];
    const long long groups = (long long)B * ((HJ + w.lt - 1) / w.lt);
    const long long need = bwd ? 3ll * sms / 2 : 3ll * sms / 4;
    if (groups >= need) return bwd ? kWalkBwd : kWalkFwd;
    return bwd ? kThreeBwd : kThreeFwd;
}

// Everything a call needs, derived from the sizes alone (no device calls).
// What a call computes besides its outputs.
enum class Mode {
    PLAIN,          // quat_cumprod_fwd / quat_cumprod_bwd
    SAVE_CARRIES,   // forward that also writes the chunk carries
    FROM_CARRIES,   // backward from caller-provided chunk carries
};

struct Plan {
    const Variant *v = nullptr;
    int vi = 0;   // index in the variant table
    qs::Geometry geo{};
    long long tiles = 0;
    int carry_lb = 32;   // lanes per block of the carry kernel
    size_t o_L = 0, o_W = 0, o_F = 0, o_H = 0, o_I = 0, ws_bytes = 0;
};

int make_plan(bool bwd, int64_t B, int64_t S, int64_t HJ, int sms, Plan *pl, Mode mode = Mode::PLAIN,
              bool bf16 = false) {
    int vi = 0;
    if (bf16) {
        int forced;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            forced = bwd ? g_bwd_variant16 : g_fwd_variant16;
        }
        if (forced >= 0) {
            vi = forced;
        } else {   // the same rule as for fp32: a walk when the lane groups fill the GPU
            const int wi = bwd ? kBwdBf16Default : kFwdBf16Default;
            const Variant &w = bwd ? kBwdBf16Variants[wi] : kFwdBf16Variants[wi];
            const long long groups = (long long)B * ((HJ + w.lt - 1) / w.lt);
            const long long need = bwd ? 3ll * sms / 2 : 3ll * sms / 4;
            vi = groups >= need ? wi : (bwd ? kBwdBf16Three : kFwdBf16Three);
        }
    } else {
        vi = pick_variant(bwd, B, HJ, sms);
    }
    const Variant *v = bf16 ? (bwd ? &kBwdBf16Variants[vi] : &kFwdBf16Variants[vi])
                            : bwd ? &kBwdVariants[vi] : &kFwdVariants[vi];
    if (mode != Mode::PLAIN && v->chain) {   // carries come from the other designs
        vi = kThreeFwd;
        v = &kFwdVariants[vi];
    }
    if (mode != Mode::PLAIN && v->T() != QS_CARRY_STEPS) {
        // The carries are defined on QS_CARRY_STEPS-step chunks: keep the
        // design, take its default configuration (which has that chunk).
        vi = v->walk ? (bwd ? kWalkBwd : kWalkFwd) : (bwd ? kThreeBwd : kThreeFwd);
        v = bwd ? &kBwdVariants[vi] : &kFwdVariants[vi];
    }
    if (mode == Mode::FROM_CARRIES && v->walk) v = &kBwdGiven;
    pl->vi = vi;
    pl->v = v;
    const int LT = pl->v->lt, T = pl->v->T();
    qs::Geometry &g = pl->geo;
    g.S = S;
    g.HJ = (int)HJ;
    g.NGb = (int)((HJ + LT - 1) / LT);
    const long long NG = (long long)B * g.NGb;
    const long long C = (S + T - 1) / T;
    pl->tiles = NG * C;
    if (NG * LT >= (1ll << 31) || pl->tiles >= (1ll << 31)) return QS_ERR_DIMS;
    g.NG = (int)NG;
    g.C = (int)C;
    g.NL = (int)(NG * LT);
    const size_t per = (size_t)pl->tiles * LT * 16;
    size_t off = sizeof(qs::WsHeader);
    if (pl->v->chain) {
        // Chained scan: status block, then per tile and lane the chunk product
        // and the inclusive value (the status words live apart, see chain_flags).
        pl->o_L = (size_t)pl->tiles * LT * 4;   // bytes of status words (their own allocation)
        pl->o_W = off;   // chunk products
        off = align_up(off + per, 256);
        pl->o_F = off;   // inclusive values
        off = align_up(off + per, 256);
        pl->ws_bytes = off;
        return QS_OK;
    }
    if (pl->v->walk) {
        // Walk kernels: status block, then (backward) the carries F_c.
        if (bwd && mode != Mode::FROM_CARRIES) {
            pl->o_F = off;
            off = align_up(off + per, 256);
        }
        pl->ws_bytes = off;
        return QS_OK;
    }
    // More threads per lane when the chunk count is large.
    pl->carry_lb = C > 256 ? 8 : 32;
    pl->o_L = off;
    off = align_up(off + per, 256);
    pl->o_F = off;
    off = align_up(off + per, 256);
    if (bwd) {
        pl->o_W = off;
        off = align_up(off + per, 256);
        pl->o_H = off;
        off = align_up(off + per, 256);
    }
    if (mode == Mode::FROM_CARRIES) {   // init = carries[:, 0], made contiguous
        pl->o_I = off;
        off = align_up(off + (size_t)B * HJ * 16, 256);
    }
    pl->ws_bytes = off;
    return QS_OK;
}

// `carries`: written (Mode::SAVE_CARRIES) or read (Mode::FROM_CARRIES),
// [B, ceil(S / QS_CARRY_STEPS), H*J] float4; unused otherwise.
// `bf16`: the tensors hold bfloat16 quaternions (8 bytes); walk kernels only.
int launch(bool bwd, const void *q, const void *d_cum, void *out, const void *init, void *d_init, int64_t B,
           int64_t S, int64_t HJ, cudaStream_t stream, Mode mode = Mode::PLAIN, float *carries = nullptr,
           bool bf16 = false) {
    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;
    Plan pl;
    rc = make_plan(bwd, B, S, HJ, di->sms, &pl, mode, bf16);
    if (rc != QS_OK) return rc;
    unsigned char *ws = nullptr;
    rc = ensure_workspace(dev, stream, pl.ws_bytes, &ws);
    if (rc != QS_OK) return rc;
    CUtensorMap qmap, dmap;
    const int eb = bf16 ? 8 : 16;
    rc = make_map(&qmap, q, B, S, HJ, pl.v->lt, pl.v->T(), eb);
    if (rc == QS_OK) rc = make_map(&dmap, bwd ? d_cum : q, B, S, HJ, pl.v->lt, pl.v->T(), eb);
    if (rc != QS_OK) return rc;
    if (pl.v->chain) {
        uint32_t epoch = 0, *flags = nullptr;
        rc = chain_flags(dev, stream, pl.o_L, &flags, &epoch);
        if (rc != QS_OK) return rc;
        qs::Control ctl;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            ctl.timeout_ns = g_timeout_ns;
            ctl.stall_tile = g_stall_tile;
        }
        ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
        const void *init4 = init;
        void *out4 = out;
        float4 *aggv = reinterpret_cast<float4 *>(ws + pl.o_W);
        float4 *inclv = reinterpret_cast<float4 *>(ws + pl.o_F);
        void *args[] = {&qmap, &init4, &out4, &flags, &aggv, &inclv, &pl.geo, &ctl, &epoch};
        if (cudaLaunchKernel(pl.v->agg, dim3((unsigned)pl.tiles), dim3(NTHREADS), args, pl.v->smem(), stream) !=
            cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        return QS_OK;
    }
    if (pl.v->walk) {
        float4 *carF = bwd ? reinterpret_cast<float4 *>(ws + pl.o_F) : nullptr;
        qs::Control ctl;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            ctl.timeout_ns = g_timeout_ns;
            ctl.stall_tile = g_stall_tile;
        }
        ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
        const void *init4 = init;   // element type of the kernel's I/O
        void *dinit4 = d_init;
        void *out4 = out;
        float4 *save4 = mode == Mode::SAVE_CARRIES ? reinterpret_cast<float4 *>(carries) : nullptr;
        const float4 *given4 = mode == Mode::FROM_CARRIES ? reinterpret_cast<const float4 *>(carries) : nullptr;
        void *fwd_args[] = {&qmap, &init4, &out4, &save4, &pl.geo, &ctl};
        void *bwd_args[] = {&qmap, &dmap, &init4, &carF, &given4, &out4, &dinit4, &pl.geo, &ctl};
        if (cudaLaunchKernel(pl.v->agg, dim3((unsigned)pl.geo.NG), dim3(pl.v->threads()),
                             bwd ? bwd_args : fwd_args, pl.v->smem(), stream) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        return QS_OK;
    }
    float4 *aggL = reinterpret_cast<float4 *>(ws + pl.o_L);
    float4 *carF = reinterpret_cast<float4 *>(ws + pl.o_F);
    float4 *aggW = bwd ? reinterpret_cast<float4 *>(ws + pl.o_W) : nullptr;
    float4 *carH = bwd ? reinterpret_cast<float4 *>(ws + pl.o_H) : nullptr;
    qs::Control ctl;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ctl.timeout_ns = g_timeout_ns;
        ctl.stall_tile = g_stall_tile;
    }
    ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
    const float4 *init4 = reinterpret_cast<const float4 *>(init);
    if (mode == Mode::FROM_CARRIES) {
        // init = carries[:, 0]: one row of H*J quaternions per batch entry.
        const size_t row = (size_t)HJ * 16;
        if (cudaMemcpy2DAsync(ws + pl.o_I, row, carries, row * pl.geo.C, row, (size_t)B, cudaMemcpyDeviceToDevice,
                              stream) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        init4 = reinterpret_cast<const float4 *>(ws + pl.o_I);
    }
    float4 *dinit4 = reinterpret_cast<float4 *>(d_init);
    float4 *out4 = reinterpret_cast<float4 *>(out);
    const float4 *aggL_c = aggL, *aggW_c = aggW, *carF_c = carF, *carH_c = carH;
    const int tiles = (int)pl.tiles;
    int lt = pl.v->lt;
    const void *carry_fn;
    // Many chunks per lane: one block per lane and a scan over 256 ranges.
    const bool scan = pl.geo.C > 256;
    if (scan) {
        carry_fn = bf16 ? (bwd ? reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoBF16, true>)
                               : reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoBF16, false>))
                        : (bwd ? reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoF32, true>)
                               : reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoF32, false>));
    } else if (bf16) {
        if (pl.carry_lb == 8)
            carry_fn = bwd ? reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoBF16, true, 8>)
                           : reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoBF16, false, 8>);
        else
            carry_fn = bwd ? reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoBF16, true, 32>)
                           : reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoBF16, false, 32>);
    } else if (pl.carry_lb == 8) {
        carry_fn = bwd ? reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoF32, true, 8>)
                       : reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoF32, false, 8>);
    } else {
        carry_fn = bwd ? reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoF32, true, 32>)
                       : reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoF32, false, 32>);
    }
    void *agg_args[] = {&qmap, &dmap, &aggL, &aggW, &pl.geo, &ctl};
    void *carry_args[] = {&aggL_c, &aggW_c, &init4, &carF, &carH, &dinit4, &pl.geo, &lt};
    void *apply_args[] = {&qmap, &dmap, &carF_c, &carH_c, &out4, &pl.geo, &ctl};
    const int carry_blocks = scan ? pl.geo.NL : (pl.geo.NL + pl.carry_lb - 1) / pl.carry_lb;
    if (cudaLaunchKernel(pl.v->agg, dim3(tiles), dim3(NTHREADS), agg_args, pl.v->smem(), stream) != cudaSuccess ||
        cudaLaunchKernel(carry_fn, dim3(carry_blocks), dim3(NTHREADS), carry_args, 0, stream) != cudaSuccess ||
        cudaLaunchKernel(pl.v->apply, dim3(tiles), dim3(NTHREADS), apply_args, pl.v->smem(), stream) !=
            cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    if (mode == Mode::SAVE_CARRIES) {
        long long total = (long long)B * pl.geo.C * HJ;
        float4 *dst = reinterpret_cast<float4 *>(carries);
        void *exp_args[] = {&carF_c, &dst, &pl.geo, &lt, &total};
        const unsigned blocks = (unsigned)((total + NTHREADS - 1) / NTHREADS);
        if (cudaLaunchKernel(reinterpret_cast<const void *>(qs::quat_export_carries_kernel), dim3(blocks),
                             dim3(NTHREADS), exp_args, 0, stream) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
    }
    return QS_OK;
}

}  // namespace

extern "C" int quat_cumprod_fwd(const float *q, const float *init, float *cum, int64_t B, int64_t S, int64_t H,
                                int64_t J, void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc == 1) return QS_OK;
    if (dc != QS_OK) return dc;
    if (!q || !init || !cum) return QS_ERR_NULL;
    if (misaligned(q) || misaligned(init) || misaligned(cum)) return QS_ERR_MISALIGNED;
    const int64_t HJ = H * J;
    const size_t big = (size_t)B * S * HJ * 16, small = (size_t)B * HJ * 16;
    if (overlaps(cum, big, q, big) || overlaps(cum, big, init, small)) return QS_ERR_ALIAS;
    return launch(false, q, nullptr, cum, init, nullptr, B, S, HJ, static_cast<cudaStream_t>(stream_));
}

extern "C" int quat_cumprod_bwd(const float *q, const float *init, const float *d_cum, float *d_q, float *d_init,
                                int64_t B, int64_t S, int64_t H, int64_t J, void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc != QS_OK && dc != 1) return dc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t HJ = H * J;
    if (dc == 1) {
        // No steps but some lanes: the gradient of init is zero.
        if (S == 0 && B > 0 && HJ > 0) {
            if (!d_init) return QS_ERR_NULL;
            if (misaligned(d_init)) return QS_ERR_MISALIGNED;
            if (cudaMemsetAsync(d_init, 0, (size_t)B * HJ * 16, stream) != cudaSuccess) {
                cudaGetLastError();
                return QS_ERR_CUDA;
            }
        }
        return QS_OK;
    }
    if (!q || !init || !d_cum || !d_q || !d_init) return QS_ERR_NULL;
    if (misaligned(q) || misaligned(init) || misaligned(d_cum) || misaligned(d_q) || misaligned(d_init))
        return QS_ERR_MISALIGNED;
    const size_t big = (size_t)B * S * HJ * 16, small = (size_t)B * HJ * 16;
    if (overlaps(d_q, big, q, big) || overlaps(d_q, big, init, small) || overlaps(d_q, big, d_cum, big) ||
        overlaps(d_init, small, q, big) || overlaps(d_init, small, init, small) ||
        overlaps(d_init, small, d_cum, big) || overlaps(d_q, big, d_init, small))
        return QS_ERR_ALIAS;
    return launch(true, q, d_cum, d_q, init, d_init, B, S, HJ, stream);
}

extern "C" int quat_cumprod_fwd_carries(const float *q, const float *init, float *cum, float *carries, int64_t B,
                                        int64_t S, int64_t H, int64_t J, void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc == 1) return QS_OK;
    if (dc != QS_OK) return dc;
    if (!q || !init || !cum || !carries) return QS_ERR_NULL;
    if (misaligned(q) || misaligned(init) || misaligned(cum) || misaligned(carries)) return QS_ERR_MISALIGNED;
    const int64_t HJ = H * J;
    const size_t big = (size_t)B * S * HJ * 16, small = (size_t)B * HJ * 16;
    const size_t ncar = (size_t)B * ((S + QS_CARRY_STEPS - 1) / QS_CARRY_STEPS) * HJ * 16;
    if (overlaps(cum, big, q, big) || overlaps(cum, big, init, small) || overlaps(carries, ncar, q, big) ||
        overlaps(carries, ncar, init, small) || overlaps(carries, ncar, cum, big))
        return QS_ERR_ALIAS;
    return launch(false, q, nullptr, cum, init, nullptr, B, S, HJ, static_cast<cudaStream_t>(stream_),
                  Mode::SAVE_CARRIES, carries);
}

extern "C" int quat_cumprod_bwd_carries(const float *q, const float *carries, const float *d_cum, float *d_q,
                                        float *d_init, int64_t B, int64_t S, int64_t H, int64_t J, void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc != QS_OK && dc != 1) return dc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t HJ = H * J;
    if (dc == 1) {
        if (S == 0 && B > 0 && HJ > 0) {   // no steps: the gradient of init is zero
            if (!d_init) return QS_ERR_NULL;
            if (misaligned(d_init)) return QS_ERR_MISALIGNED;
            if (cudaMemsetAsync(d_init, 0, (size_t)B * HJ * 16, stream) != cudaSuccess) {
                cudaGetLastError();
                return QS_ERR_CUDA;
            }
        }
        return QS_OK;
    }
    if (!q || !carries || !d_cum || !d_q || !d_init) return QS_ERR_NULL;
    if (misaligned(q) || misaligned(carries) || misaligned(d_cum) || misaligned(d_q) || misaligned(d_init))
        return QS_ERR_MISALIGNED;
    const size_t big = (size_t)B * S * HJ * 16, small = (size_t)B * HJ * 16;
    const size_t ncar = (size_t)B * ((S + QS_CARRY_STEPS - 1) / QS_CARRY_STEPS) * HJ * 16;
    if (overlaps(d_q, big, q, big) || overlaps(d_q, big, carries, ncar) || overlaps(d_q, big, d_cum, big) ||
        overlaps(d_init, small, q, big) || overlaps(d_init, small, carries, ncar) ||
        overlaps(d_init, small, d_cum, big) || overlaps(d_q, big, d_init, small))
        return QS_ERR_ALIAS;
    return launch(true, q, d_cum, d_q, nullptr, d_init, B, S, HJ, stream, Mode::FROM_CARRIES,
                  const_cast<float *>(carries));
}

extern "C" int quat_cumprod_fwd_bf16(const uint16_t *q, const uint16_t *init, uint16_t *cum, int64_t B, int64_t S,
                                     int64_t H, int64_t J, void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc == 1) return QS_OK;
    if (dc != QS_OK) return dc;
    const int64_t HJ = H * J;
    if (HJ % 2 != 0) return QS_ERR_DIMS;   // TMA row strides are multiples of 16 bytes
    if (!q || !init || !cum) return QS_ERR_NULL;
    if (misaligned(q) || misaligned(init) || misaligned(cum)) return QS_ERR_MISALIGNED;
    const size_t big = (size_t)B * S * HJ * 8, small = (size_t)B * HJ * 8;
    if (overlaps(cum, big, q, big) || overlaps(cum, big, init, small)) return QS_ERR_ALIAS;
    return launch(false, q, nullptr, cum, init, nullptr, B, S, HJ, static_cast<cudaStream_t>(stream_), Mode::PLAIN,
                  nullptr, true);
}

extern "C" int quat_cumprod_bwd_bf16(const uint16_t *q, const uint16_t *init, const uint16_t *d_cum,
                                     uint16_t *d_q, uint16_t *d_init, int64_t B, int64_t S, int64_t H, int64_t J,
                                     void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc != QS_OK && dc != 1) return dc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t HJ = H * J;
    if (dc == 1) {
        if (S == 0 && B > 0 && HJ > 0) {   // no steps: the gradient of init is zero
            if (!d_init) return QS_ERR_NULL;
            if (misaligned(d_init)) return QS_ERR_MISALIGNED;
            if (cudaMemsetAsync(d_init, 0, (size_t)B * HJ * 8, stream) != cudaSuccess) {
                cudaGetLastError();
                return QS_ERR_CUDA;
            }
        }
        return QS_OK;
    }
    if (HJ % 2 != 0) return QS_ERR_DIMS;
    if (!q || !init || !d_cum || !d_q || !d_init) return QS_ERR_NULL;
    if (misaligned(q) || misaligned(init) || misaligned(d_cum) || misaligned(d_q) || misaligned(d_init))
        return QS_ERR_MISALIGNED;
    const size_t big = (size_t)B * S * HJ * 8, small = (size_t)B * HJ * 8;
    if (overlaps(d_q, big, q, big) || overlaps(d_q, big, init, small) || overlaps(d_q, big, d_cum, big) ||
        overlaps(d_init, small, q, big) || overlaps(d_init, small, init, small) ||
        overlaps(d_init, small, d_cum, big) || overlaps(d_q, big, d_init, small))
        return QS_ERR_ALIAS;
    return launch(true, q, d_cum, d_q, init, d_init, B, S, HJ, stream, Mode::PLAIN, nullptr, true);
}

extern "C" int quat_cumprod_status(void *stream_) {
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    unsigned char *base = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_ws.find({dev, reinterpret_cast<uintptr_t>(stream)});
        if (it == g_ws.end() || !it->second.base) return QS_OK;
        base = it->second.base;
    }
    qs::WsHeader h;
    if (cudaMemcpy(&h, base, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    if (h.err_code == 0) return QS_OK;
    if (cudaMemset(base, 0, sizeof(qs::WsHeader)) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    return QS_ERR_TIMEOUT;
}

extern "C" int quat_cumprod_plan(int call, int64_t B, int64_t S, int64_t H, int64_t J, int *variant, int *kernels) {
    if (!variant || !kernels) return QS_ERR_NULL;
    if (call < 0 || call > 5) return QS_ERR_DIMS;
    const bool bwd = (call & 1) != 0;
    const bool bf16 = call >= 4;
    const Mode mode = call == 2 ? Mode::SAVE_CARRIES : call == 3 ? Mode::FROM_CARRIES : Mode::PLAIN;
    if (bf16 && (H * J) % 2 != 0 && B > 0 && S > 0 && H > 0 && J > 0) return QS_ERR_DIMS;
    const int dc = check_dims(B, S, H, J);
    if (dc != QS_OK && dc != 1) return dc;
    if (dc == 1) {   // nothing to launch (the backward may write d_init with a memset)
        *variant = -1;
        *kernels = 0;
        return QS_OK;
    }
    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;
    Plan pl;
    rc = make_plan(bwd, B, S, H * J, di->sms, &pl, mode, bf16);
    if (rc != QS_OK) return rc;
    *variant = pl.vi;
    *kernels = (pl.v->walk || pl.v->chain) ? 1 : (mode == Mode::SAVE_CARRIES ? 4 : 3);
    return QS_OK;
}

extern "C" const char *quat_cumprod_strerror(int status) {
    switch (status) {
        case QS_OK: return "success";
        case QS_ERR_NULL: return "a required pointer is NULL";
        case QS_ERR_DIMS: return "a size is negative or beyond the supported limits";
        case QS_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
        case QS_ERR_ALIAS: return "an output overlaps an input";
        case QS_ERR_CUDA: return "a CUDA runtime call failed";
        case QS_ERR_TIMEOUT: return "a device-side wait ran out (outputs are invalid)";
        case QS_ERR_NOMEM: return "workspace allocation failed or would be needed during stream capture";
        case QS_ERR_DEVICE: return "the current device is not compute capability 10.3 (sm_103)";
        case QS_ERR_SCRATCH:
            return "the sizes need more scratch than quat_cumprod_bwd_noalloc's fixed array holds "
                   "(B * ceil(H*J/32) * ceil(S/64) must not exceed QS_NOALLOC_MAX_TILES = 8192)";
        default: return "unknown status";
    }
}

extern "C" int quat_cumprod_debug_set_timeout_ns(int64_t ns) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_timeout_ns = ns > 0 ? (unsigned long long)ns : DEFAULT_TIMEOUT_NS;
    return QS_OK;
}

extern "C" int quat_cumprod_debug_stall_tile(int64_t tile) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_stall_tile = (tile < 0 || tile > INT32_MAX) ? -1 : (int)tile;
    return QS_OK;
}

extern "C" int quat_cumprod_debug_set_variant_bf16(int fwd_variant, int bwd_variant) {
    if (fwd_variant >= kNumFwdBf16 || bwd_variant >= kNumBwdBf16) return QS_ERR_DIMS;
    std::lock_guard<std::mutex> lk(g_mu);
    g_fwd_variant16 = fwd_variant < 0 ? -1 : fwd_variant;
    g_bwd_variant16 = bwd_variant < 0 ? -1 : bwd_variant;
    return QS_OK;
}

extern "C" int quat_cumprod_debug_set_variant(int fwd_variant, int bwd_variant) {
    if (fwd_variant >= kNumFwd || bwd_variant >= kNumBwd) return QS_ERR_DIMS;
    std::lock_guard<std::mutex> lk(g_mu);
    g_fwd_variant = fwd_variant < 0 ? -1 : fwd_variant;
    g_bwd_variant = bwd_variant < 0 ? -1 : bwd_variant;
    return QS_OK;
}

// ===========================================================================
// quat_cumprod_bwd_noalloc: the backward of quat_cumprod_bwd with its scratch
// (status block, chunk aggregates and carries) in one fixed device array of
// this file instead of the cudaMalloc'ed per-stream workspace.  Same kernels,
// always the 32-lane x 64-step tile, so that the size limit is fixed too.
// ===========================================================================
namespace {

constexpr int NA_LT = 32, NA_N = 8;
constexpr int NA_T = (NTHREADS / NA_LT) * NA_N;                                  // 64 steps per chunk
constexpr size_t NA_ARRAY_BYTES = size_t(QS_NOALLOC_MAX_TILES) * NA_LT * 16;   // one aggregate or carry array
constexpr size_t NA_SCRATCH_BYTES = sizeof(qs::WsHeader) + 4 * NA_ARRAY_BYTES;
static_assert(sizeof(qs::WsHeader) == 256, "the arrays after the status block stay 256-byte aligned");
static_assert(NA_SCRATCH_BYTES == (size_t(16) << 20) + 256, "the header states 16 MiB + 256 bytes");

}  // namespace

// The scratch every quat_cumprod_bwd_noalloc call on a device shares (one copy
// per device, like every __device__ variable).
static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_SCRATCH_BYTES];

namespace {

std::map<int, unsigned char *> g_noalloc_ptr;   // device -> address of g_noalloc_scratch

// Address of the scratch on the current device `dev`, looked up once per
// device (the lookup loads this library's device code on that device).
int noalloc_scratch(int dev, unsigned char **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_noalloc_ptr.find(dev);
    if (it != g_noalloc_ptr.end()) {
        *out = it->second;
        return QS_OK;
    }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<unsigned char *>(p);
    *out = static_cast<unsigned char *>(p);
    return QS_OK;
}

// Work tiles of the fixed tile for these sizes (exact; no overflow for any
// sizes that passed check_dims).
long long noalloc_tiles(int64_t B, int64_t S, int64_t HJ) {
    const __int128 t = (__int128)B * ((HJ + NA_LT - 1) / NA_LT) * ((S + NA_T - 1) / NA_T);
    return t > (__int128)INT64_MAX ? INT64_MAX : (long long)t;
}

int noalloc_launch(const float *q, const float *init, const float *d_cum, float *d_q, float *d_init, int64_t B,
                   int64_t S, int64_t HJ, cudaStream_t stream) {
    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;
    unsigned char *ws = nullptr;
    rc = noalloc_scratch(dev, &ws);
    if (rc != QS_OK) return rc;

    qs::Geometry geo;
    geo.S = S;
    geo.HJ = (int)HJ;
    geo.NGb = (int)((HJ + NA_LT - 1) / NA_LT);
    geo.NG = (int)(B * geo.NGb);
    geo.C = (int)((S + NA_T - 1) / NA_T);
    geo.NL = geo.NG * NA_LT;
    const int tiles = geo.NG * geo.C;
    const size_t per = (size_t)tiles * NA_LT * 16;
    float4 *aggL = reinterpret_cast<float4 *>(ws + sizeof(qs::WsHeader));
    float4 *carF = aggL + per / 16;
    float4 *aggW = carF + per / 16;
    float4 *carH = aggW + per / 16;

    // The status block must start at zero; every aggregate and carry slot a
    // call reads is written earlier in the same call.
    if (cudaMemsetAsync(ws, 0, sizeof(qs::WsHeader), stream) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    CUtensorMap qmap, dmap;
    rc = make_map(&qmap, q, B, S, HJ, NA_LT, NA_T);
    if (rc == QS_OK) rc = make_map(&dmap, d_cum, B, S, HJ, NA_LT, NA_T);
    if (rc != QS_OK) return rc;
    qs::Control ctl;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ctl.timeout_ns = g_timeout_ns;
    }
    ctl.stall_tile = -1;
    ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
    const float4 *init4 = reinterpret_cast<const float4 *>(init);
    float4 *dinit4 = reinterpret_cast<float4 *>(d_init);
    float4 *out4 = reinterpret_cast<float4 *>(d_q);
    const float4 *aggL_c = aggL, *aggW_c = aggW, *carF_c = carF, *carH_c = carH;
    int lt = NA_LT;
    const int carry_lb = geo.C > 256 ? 8 : 32;
    const void *agg_fn = reinterpret_cast<const void *>(qs::quat_agg_kernel<qs::IoF32, true, NA_LT, NA_N>);
    const void *apply_fn = reinterpret_cast<const void *>(qs::quat_apply_kernel<qs::IoF32, true, NA_LT, NA_N>);
    const void *carry_fn = carry_lb == 8 ? reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoF32, true, 8>)
                                         : reinterpret_cast<const void *>(qs::quat_carry_kernel<qs::IoF32, true, 32>);
    const size_t smem = qs::tile_smem_bytes(true, NA_LT, NA_N);
    void *agg_args[] = {&qmap, &dmap, &aggL, &aggW, &geo, &ctl};
    void *carry_args[] = {&aggL_c, &aggW_c, &init4, &carF, &carH, &dinit4, &geo, &lt};
    void *apply_args[] = {&qmap, &dmap, &carF_c, &carH_c, &out4, &geo, &ctl};
    const int carry_blocks = (geo.NL + carry_lb - 1) / carry_lb;
    if (cudaLaunchKernel(agg_fn, dim3(tiles), dim3(NTHREADS), agg_args, smem, stream) != cudaSuccess ||
        cudaLaunchKernel(carry_fn, dim3(carry_blocks), dim3(NTHREADS), carry_args, 0, stream) != cudaSuccess ||
        cudaLaunchKernel(apply_fn, dim3(tiles), dim3(NTHREADS), apply_args, smem, stream) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    return QS_OK;
}

}  // namespace

extern "C" int quat_cumprod_bwd_noalloc(const float *q, const float *init, const float *d_cum, float *d_q,
                                        float *d_init, int64_t B, int64_t S, int64_t H, int64_t J, void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc != QS_OK && dc != 1) return dc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t HJ = H * J;
    if (dc == 1) {
        if (S == 0 && B > 0 && HJ > 0) {   // no steps: the gradient of init is zero
            if (!d_init) return QS_ERR_NULL;
            if (misaligned(d_init)) return QS_ERR_MISALIGNED;
            if (cudaMemsetAsync(d_init, 0, (size_t)B * HJ * 16, stream) != cudaSuccess) {
                cudaGetLastError();
                return QS_ERR_CUDA;
            }
        }
        return QS_OK;
    }
    if (!q || !init || !d_cum || !d_q || !d_init) return QS_ERR_NULL;
    if (misaligned(q) || misaligned(init) || misaligned(d_cum) || misaligned(d_q) || misaligned(d_init))
        return QS_ERR_MISALIGNED;
    const size_t big = (size_t)B * S * HJ * 16, small = (size_t)B * HJ * 16;
    if (overlaps(d_q, big, q, big) || overlaps(d_q, big, init, small) || overlaps(d_q, big, d_cum, big) ||
        overlaps(d_init, small, q, big) || overlaps(d_init, small, init, small) ||
        overlaps(d_init, small, d_cum, big) || overlaps(d_q, big, d_init, small))
        return QS_ERR_ALIAS;
    if (noalloc_tiles(B, S, HJ) > QS_NOALLOC_MAX_TILES) return QS_ERR_SCRATCH;
    return noalloc_launch(q, init, d_cum, d_q, d_init, B, S, HJ, stream);
}
