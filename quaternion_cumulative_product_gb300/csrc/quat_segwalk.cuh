// quat_segwalk.cuh -- the segmented chained walk (forward): persistent CTAs,
// each unit one lane group over a segment of K chunks, segments chained by
// decoupled look-back.
#pragma once

#include "quat_chain.cuh"   // status words of the look-back
#include "quat_walk.cuh"    // bounded ring waits

namespace qs {

// ---------------------------------------------------------------------------
// Segmented chained walk.  The sequence of each lane group is cut into
// segments of K chunks; unit u = (segment p, lane group g) with u = p*NG + g,
// so every lane group's segment p comes before any segment p+1.  Persistent
// CTAs take units in that order from a ticket counter, so a unit waits only on
// units already taken by running CTAs.  Per unit:
//
//   1. walk the segment's chunks (q loaded with the L2 evict-last policy) and
//      fold the chunk products into the segment product A;
//   2. publish A, look back over the lane group's earlier segments (their
//      products, back to the nearest published inclusive value) for the
//      carry X entering the segment, publish the inclusive value A (x) X;
//   3. walk the segment again, now from L2 (evict-first), and write
//      cum[t] = (local product) (x) X chunk by chunk.
//
// DRAM traffic is one read of q and one write of cum (32 bytes per element)
// as long as the segments in flight fit in L2, and the look-back is paid once
// per segment instead of once per chunk.  The chunks of one CTA's units, both
// walks, form one item sequence through a single TMA ring: the producer
// thread (one that never folds) runs NST items ahead, across unit
// boundaries, taking the next unit's ticket when its cursor gets there, so the
// look-back of a unit overlaps the loads of its second walk.
//
// Tickets: ctr[0] counts the units taken, ctr[1] the CTAs that finished; the
// last CTA to finish sets both back to zero, so every launch starts from zero
// (every wait is bounded, so every CTA finishes).  Status words of the
// look-back are those of the chained scan (epoch << 2 | CH_AGG / CH_INCL),
// one per lane and unit.  A unit whose wait ran out still publishes (NaN).
// ---------------------------------------------------------------------------

// A value the look-back reads is published once none of its four words holds
// the all-ones pattern the arrays are reset to before each launch (SENT);
// arithmetic never yields that pattern (a NaN result is the canonical one).
__device__ __forceinline__ bool lb_published(const float4 v) {
    return __float_as_uint(v.x) != 0xffffffffu && __float_as_uint(v.y) != 0xffffffffu &&
           __float_as_uint(v.z) != 0xffffffffu && __float_as_uint(v.w) != 0xffffffffu;
}

// SENT: the segment products and inclusive values carry their own state: a
// launch reads buffers (agg, incl) that hold all-ones bits wherever nothing is
// published yet, so a look-back round loads the predecessors' products and
// inclusive values together (one memory latency) and the status words go
// unused.  Each unit, once published, resets its entries of the other pair of
// buffers (agg_next, incl_next), which the next launch reads; if a wait ran
// out and units were left undone, the last CTA resets all of them.  Otherwise
// the values are published behind epoch-tagged status words (two latencies
// per round) and agg_next / incl_next are unused.
__device__ __forceinline__ float4 lb_unpublished() {
    const float n = __uint_as_float(0xffffffffu);
    return make_float4(n, n, n, n);
}

// `carries` (may be null): [B, C, H*J] float4, the state entering every
// chunk, carries[b, c] = cum[b, c*T - 1] (init for c = 0).
template <typename IO, int LT, int NSEG, int N, int NST, int K, bool SENT = false>
__global__ void __launch_bounds__(LT *NSEG)
    quat_segwalk_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const typename IO::elem *__restrict__ init,
                            typename IO::elem *__restrict__ out, float4 *__restrict__ carries,
                            uint32_t *__restrict__ flags,
                            unsigned int *__restrict__ ctr, float4 *__restrict__ agg,
                            float4 *__restrict__ incl, float4 *__restrict__ agg_next, float4 *__restrict__ incl_next,
                            const Geometry geo, const Control ctl, uint32_t epoch) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr int NT = LT * NSEG;
    constexpr uint32_t BYTES = T * LT * IO::bytes;
    constexpr int NU = 8;   // unit slots: the producer is at most NST items (>= NST / 2 units) ahead
    static_assert(NST / 2 + 2 <= NU, "unit slots");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    __shared__ __align__(8) uint64_t full[NST];
    __shared__ int issued[NST];
    __shared__ int s_broken;
    __shared__ int s_unit[NU];              // ticket of the CTA's k-th unit (slot k % NU), -1: no more
    __shared__ float4 s_a[2][NSEG][LT];     // segment products of item i (slot i & 1)
    __shared__ float4 s_x[2][LT];           // carry into item i of the second walk (slot i & 1)
    __shared__ float4 s_lb[NSEG][LT];       // one look-back round: a partial product per segment
    __shared__ uint32_t s_st[NSEG][LT];

    const int tid = static_cast<int>(threadIdx.x);
    const int lane = tid % LT, seg = tid / LT;
    const int NG = geo.NG, C = geo.C;
    const int P = (C + K - 1) / K;
    const int U = P * NG;
    constexpr int kWarp1 = (LT + 31) / 32 * 32;   // producer: first thread of the first warp without segment 0
    const bool producer = tid == (kWarp1 < NT ? kWarp1 : NT - 1);

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            issued[s] = 0;
        }
        for (int u = 0; u < NU; ++u) s_unit[u] = -1;
        fence_mbar_init();
        s_broken = 0;
    }
    __syncthreads();
    const uint64_t keep = l2_policy_evict_last();
    const uint64_t drop = l2_policy_evict_first();

    // ---- producer cursor (registers of the producer thread) -------------------
    int pk = 0;          // CTA-local unit number the cursor is in
    int pj = 0;          // item within that unit (0 .. 2n-1)
    int pn = 0;          // items of that unit, 0: unit not taken yet
    int pt = 0;          // its ticket
    bool pend = false;   // no more units
    int pit = 0;         // items issued
    auto issue_next = [&]() {
        if (pend) return;
        if (pn == 0) {   // enter unit pk: take its ticket
            const int t = static_cast<int>(atomicAdd(ctr, 1u));
            if (t >= U) {
                pend = true;
                s_unit[pk % NU] = -1;
                return;
            }
            pt = t;
            s_unit[pk % NU] = t;
            const int p = t / NG;
            pn = 2 * min(K, C - p * K);
            pj = 0;
        }
        const int p = pt / NG, g = pt - p * NG;
        const int b = g / geo.NGb, x0 = (g - b * geo.NGb) * LT * 4;
        const bool first = pj < pn / 2;
        const int c = p * K + (first ? pj : pj - pn / 2);
        const int st = pit % NST;
        ++issued[st];
        mbar_arrive_expect_tx(&full[st], BYTES + (first && c * NG + g == ctl.stall_tile ? 16u : 0u));
        tma_load_3d_hint(ring + st * BYTES, &qmap, x0, c * T, b, &full[st], first ? keep : drop);
        ++pit;
        if (++pj == pn) {
            ++pk;
            pn = 0;
        }
    };
    if (producer)
        for (int i = 0; i < NST; ++i) issue_next();
    __syncthreads();

    const uint32_t tag = epoch << 2;
    int it = 0;   // items consumed (every thread)
    for (int k = 0;; ++k) {
        // A slot the producer has not filled reads -1: after a wait ran out
        // the producer takes no more units, and the CTA ends with the units
        // it already took (walked without waiting, still published).
        const int t = s_unit[k % NU];
        if (t < 0) break;
        const int p = t / NG, g = t - p * NG;
        const int b = g / geo.NGb;
        const int hj = (g - b * geo.NGb) * LT + lane;
        const bool lane_ok = hj < geo.HJ;
        const int c0 = p * K, n = min(K, C - c0);

        // ---- 1. segment product ---------------------------------------------
        float4 A = q_ident();   // segment-0 threads
        for (int j = 0; j < n; ++j, ++it) {
            const int st = it % NST, sl = it & 1;
            const E *Qt = reinterpret_cast<const E *>(ring + st * BYTES);
            if (!ld_volatile_int(&s_broken) && !wait_stage(&full[st], (it / NST) & 1, ctl, (c0 + j) * NG + g))
                s_broken = 1;
            float4 loc = q_ident();
#pragma unroll
            for (int kk = 0; kk < N; ++kk) loc = q_mul(IO::get(Qt[(seg * N + kk) * LT + lane]), loc);
            s_a[sl][seg][lane] = loc;
            __syncthreads();
            if (producer && !s_broken) issue_next();
            if (seg == 0) {
#pragma unroll
                for (int kk = 0; kk < NSEG; ++kk) A = q_mul(s_a[sl][kk][lane], A);
            }
        }

        // ---- 2. publish, look back, publish ------------------------------------
        const long long me = static_cast<long long>(t) * LT + lane;
        float4 acc = q_ident();
        bool done = p == 0;
        if (p == 0) {
            if (seg == 0 && lane_ok) acc = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
        } else if (seg == 0) {   // the product first: later segments can use it before the carry is known
            __stcg(agg + me, A);
            if constexpr (!SENT) st_release_u32(flags + me, tag | CH_AGG);
        }
        // acc = A_{p-1} (x) A_{p-2} (x) ... (x) incl.  Per round the NSEG
        // segment threads of a lane take LB predecessors each (segment k:
        // segments base - k*LB .. base - k*LB - LB + 1), load their LB status
        // words together, then the values up to the first inclusive one
        // together, and fold them; segment 0 combines the partial products in
        // order.  Two memory latencies per round of NSEG * LB predecessors.
        constexpr int LB = 4;
        if (p > 0) {
            for (int base = p - 1;; base -= NSEG * LB) {
                float4 part = q_ident();
                uint32_t pst = 0;   // CH_INCL once the fold reached an inclusive value
                if constexpr (SENT) {
                    float4 av[LB], iv[LB];
                    long long idx[LB];
                    bool real[LB];
#pragma unroll
                    for (int j = 0; j < LB; ++j) {   // products and inclusive values, loaded together
                        const int pp = base - seg * LB - j;
                        real[j] = pp >= 0;
                        idx[j] = (static_cast<long long>(pp < 0 ? 0 : pp) * NG + g) * LT + lane;
                        av[j] = q_ident();
                        iv[j] = q_ident();   // before segment 0: an inclusive identity
                        if (real[j]) {
                            av[j] = __ldcg(agg + idx[j]);
                            iv[j] = __ldcg(incl + idx[j]);
                        }
                    }
                    bool lost = false, stop = false;
#pragma unroll
                    for (int j = 0; j < LB; ++j) {
                        if (stop) break;
                        if (real[j] && !lb_published(iv[j]) && !lb_published(av[j]) && !lost) {
                            const unsigned long long t0 = global_timer_ns();
                            do {
                                if (global_timer_ns() - t0 > ctl.timeout_ns) {
                                    record_error(ctl.hdr, c0 * NG + g);
                                    lost = true;
                                    break;
                                }
                                av[j] = __ldcg(agg + idx[j]);
                                iv[j] = __ldcg(incl + idx[j]);
                            } while (!lb_published(iv[j]) && !lb_published(av[j]));
                        }
                        if (lost) {
                            part = q_nan();
                            pst = CH_INCL;
                            stop = true;
                        } else if (!real[j] || lb_published(iv[j])) {
                            part = q_mul(part, iv[j]);
                            pst = CH_INCL;
                            stop = true;
                        } else {
                            part = q_mul(part, av[j]);
                        }
                    }
                } else {
                    uint32_t f[LB];
                    long long idx[LB];
#pragma unroll
                    for (int j = 0; j < LB; ++j) {
                        const int pp = base - seg * LB - j;
                        idx[j] = (static_cast<long long>(pp < 0 ? 0 : pp) * NG + g) * LT + lane;
                        // before segment 0 there is nothing to fold: an inclusive identity
                        f[j] = pp < 0 ? (tag | CH_INCL) : ld_acquire_u32(flags + idx[j]);
                    }
                    bool lost = false;
#pragma unroll
                    for (int j = 0; j < LB; ++j) {
                        if ((f[j] & ~3u) == tag || lost) continue;
                        const unsigned long long t0 = global_timer_ns();
                        do {
                            if (global_timer_ns() - t0 > ctl.timeout_ns) {
                                record_error(ctl.hdr, c0 * NG + g);
                                lost = true;
                                break;
                            }
                            f[j] = ld_acquire_u32(flags + idx[j]);
                        } while ((f[j] & ~3u) != tag);
                    }
                    if (lost) {
                        part = q_nan();
                        pst = CH_INCL;
                    } else {
                        float4 v[LB];
                        bool stop = false;
#pragma unroll
                        for (int j = 0; j < LB; ++j) {   // the values to fold, loaded together
                            const bool use = !stop;
                            const bool inc = (f[j] & 3u) == CH_INCL;
                            const bool real = base - seg * LB - j >= 0;
                            v[j] = q_ident();
                            if (use && real) v[j] = inc ? __ldcg(incl + idx[j]) : __ldcg(agg + idx[j]);
                            stop = stop || inc;
                        }
                        stop = false;
#pragma unroll
                        for (int j = 0; j < LB; ++j) {
                            if (stop) break;
                            part = q_mul(part, v[j]);
                            if ((f[j] & 3u) == CH_INCL) {
                                pst = CH_INCL;
                                stop = true;
                            }
                        }
                    }
                }
                s_lb[seg][lane] = part;
                s_st[seg][lane] = pst;
                __syncthreads();
                if (seg == 0 && !done) {
#pragma unroll 1
                    for (int kk = 0; kk < NSEG; ++kk) {
                        acc = q_mul(acc, s_lb[kk][lane]);
                        if (s_st[kk][lane] == CH_INCL) {
                            done = true;
                            break;
                        }
                    }
                }
                if (!__syncthreads_or(seg == 0 && !done)) break;
            }
        }
        if (seg == 0) {
            __stcg(incl + me, q_mul(A, acc));
            if constexpr (!SENT) st_release_u32(flags + me, tag | CH_INCL);
            if constexpr (SENT) {   // this unit's entries of the next launch's buffers
                __stcg(agg_next + me, lb_unpublished());
                __stcg(incl_next + me, lb_unpublished());
            }
            s_x[it & 1][lane] = acc;   // carry into the first item of the second walk
        }
        __syncthreads();

        // ---- 3. second walk: cum ---------------------------------------------
        const long long row0 = static_cast<long long>(b) * geo.S;
        float4 R = acc;   // segment-0 threads: carry into the next chunk
        for (int j = 0; j < n; ++j, ++it) {
            const int st = it % NST, sl = it & 1;
            const E *Qt = reinterpret_cast<const E *>(ring + st * BYTES);
            if (!ld_volatile_int(&s_broken) && !wait_stage(&full[st], (it / NST) & 1, ctl, (c0 + j) * NG + g))
                s_broken = 1;
            float4 x[N];
            float4 loc = q_ident();
#pragma unroll
            for (int kk = 0; kk < N; ++kk) {
                loc = q_mul(IO::get(Qt[(seg * N + kk) * LT + lane]), loc);
                x[kk] = loc;
            }
            s_a[sl][seg][lane] = loc;
            __syncthreads();
            if (producer && !s_broken) issue_next();
            float4 Pr = q_ident();   // product of the earlier segments of the chunk
#pragma unroll
            for (int kk = 0; kk < NSEG - 1; ++kk)
                if (kk < seg) Pr = q_mul(s_a[sl][kk][lane], Pr);
            const float4 Y = q_mul(Pr, s_x[sl][lane]);
            if (seg == 0) {
                if (carries != nullptr && lane_ok)   // the state entering chunk c0 + j
                    carries[(static_cast<long long>(b) * C + c0 + j) * geo.HJ + hj] = R;
                float4 L = q_ident();
#pragma unroll
                for (int kk = 0; kk < NSEG; ++kk) L = q_mul(s_a[sl][kk][lane], L);
                R = q_mul(L, R);
                s_x[sl ^ 1][lane] = R;
            }
            const long long t0 = static_cast<long long>(c0 + j) * T + seg * N;
            E *dst = out + (row0 + t0) * geo.HJ + hj;
            if (lane_ok && t0 + N <= geo.S) {
#pragma unroll
                for (int kk = 0; kk < N; ++kk)
                    __stcs(dst + static_cast<long long>(kk) * geo.HJ, IO::put(q_mul(x[kk], Y)));
            } else if (lane_ok) {
#pragma unroll
                for (int kk = 0; kk < N; ++kk)
                    if (t0 + kk < geo.S) __stcs(dst + static_cast<long long>(kk) * geo.HJ, IO::put(q_mul(x[kk], Y)));
            }
        }
        if (tid == 0) {
            s_unit[k % NU] = -1;   // (the producer is fewer than NU units ahead)
            if constexpr (SENT) atomicAdd(ctr + 2, 1u);   // units done
        }
        __syncthreads();   // the unit's shared slots are read before the next unit writes them
    }
    if (s_broken) drain_ring<NST>(full, issued, ctl);
    // The last CTA to finish resets the counters for the next launch (and,
    // SENT, the next buffers if units were left undone).
    __shared__ int s_last, s_short;
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(ctr + 1, 1u) == gridDim.x - 1;
        s_short = s_last && atomicAdd(ctr + 2, 0u) != static_cast<unsigned int>(U);
    }
    __syncthreads();
    if (s_last) {
        if (SENT && s_short) {
            const long long n = static_cast<long long>(U) * LT;
            for (long long i = tid; i < n; i += NT) {
                __stcg(agg_next + i, lb_unpublished());
                __stcg(incl_next + i, lb_unpublished());
            }
        }
        if (tid == 0) {
            atomicExch(ctr, 0u);
            atomicExch(ctr + 1, 0u);
            atomicExch(ctr + 2, 0u);
        }
    }
}

// Dynamic shared memory: the ring.
__host__ __device__ constexpr size_t segwalk_smem_bytes(int lt, int nseg, int n, int nst, int eb = 16) {
    return 128 + size_t(nst) * nseg * n * lt * eb;
}

}  // namespace qs
