// quat_chain.cuh -- the single-pass chained-scan forward (decoupled look-back).
#pragma once

#include "quat_common.cuh"

namespace qs {

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

}  // namespace qs
