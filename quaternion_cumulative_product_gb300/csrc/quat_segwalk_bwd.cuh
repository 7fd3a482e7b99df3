// quat_segwalk_bwd.cuh -- the segmented chained walk of the backward: units
// (segment, lane group) taken from the right end of the sequence, each walked
// twice, segments chained right to left by decoupled look-back over their
// affine cotangent maps.  Warp-specialised CTAs: compute warps, a producer
// warp and a look-back warp, as in quat_segwalk_ws_fwd_kernel.
#pragma once

#include "quat_segwalk_ws.cuh"

namespace qs {

// ---------------------------------------------------------------------------
// With H[t] = conj(q_t) (x) G[t], the cotangent step t hands to cum[t-1], the
// reverse recurrence G[t] = d_cum[t] + H[t+1] makes a run of steps an affine
// map of the H entering it from the right:
//
//     H_left = V + conj(A) (x) H_right,
//     A = q_{t1-1} (x) ... (x) q_{t0},   V = sum_s conj(q_s (x) ... (x) q_{t0}) (x) d_cum[s],
//
// (the page's suffix-sum factorisation conj(P_s) = conj(P_{t0-1}) (x)
// conj(local_s), exact for every quaternion).  The sequence of each lane group
// is cut into segments of K chunks counted from the right end; unit
// u = p * NG + g is segment p (p = 0 the rightmost) of lane group g, so every
// lane group's segment p comes before any segment p + 1, and a unit waits
// only on units taken earlier by running CTAs.  Per unit:
//
//   1. walk 1 (chunks left to right; q and d_cum loaded with the L2
//      evict-last policy): every compute thread writes the product and the
//      weighted sum of its N steps of each chunk into the unit's table in
//      shared memory;
//   2. the look-back warp folds the table into the unit's map (V, A),
//      publishes it, folds the maps of the segments to its right back to the
//      nearest published inclusive value into the H entering the unit from
//      the right, publishes the inclusive value H_left (d_init for the
//      leftmost segment), then replaces every table entry by the cum just
//      before that thread's steps (from the chunk's carry) and the H entering
//      them from the right;
//   3. walk 2 (chunks right to left, from L2, evict-first): each thread walks
//      its N steps from its two table entries: cum[t-1] forward, then
//      G[t] = d_cum[t] + H[t+1], d_q[t] = G[t] (x) conj(cum[t-1]),
//      H[t] = conj(q_t) (x) G[t] backward.
//
// Neither walk has a block barrier: the compute warps hand stages back and
// units on through mbarriers, and the serial folds of a unit run on the
// look-back warp while the compute warps walk the next unit.  Per element the walks take six quaternion products (two in walk 1,
// four in walk 2).
//
// The forward carries come from `carries` [B, C, H*J] (carries[b, c] =
// cum[b, c*T - 1], init for c = 0): saved by the forward, or written by the
// forward segmented walk's carries-only pass just before.  DRAM traffic is one
// read of q and d_cum and one write of d_q (48 bytes per element) as long as
// the units in flight fit in L2.
//
// Look-back values carry their own state (as the forward's SENT form): a
// launch reads buffers (V, A, incl) that hold all-ones words wherever nothing
// is published; a value counts as published once none of its words holds that
// pattern (arithmetic never yields it).  Each unit, once published, resets its
// entries of the other triple of buffers, which the next launch reads; if a
// wait ran out and units were left undone, the last CTA resets all of them.
// Tickets: ctr[0] units taken, ctr[1] CTAs finished, ctr[2] units done; the
// last CTA sets them back to zero.
// ---------------------------------------------------------------------------

// W2FWD: walk 2 takes the unit's chunks left to right, in walk 1's order (its
// chunks are independent: every thread starts from its table entries), so
// every chunk is read again the same number of items after its first read;
// otherwise right to left, starting with the chunk walk 1 read last.
// NLB: look-back warps (1 or 2); with two, unit k goes to look-back warp
// k % 2, so that one unit's look-back overlaps the previous one's.
// DL: walk 2 of unit k follows walk 1 of unit k + DL (items W1(u_k),
// W2(u_{k-DL})), so a unit's look-back has DL first walks (and DL - 1 second
// walks) of later units to finish in; DL + 1 unit slots of the tables.
template <typename IO, int LT, int NSEG, int N, int NST, int K, int MINB = 1, int LB = 4, bool W2FWD = false,
          int NLB = 1, int DL = 1>
__global__ void __launch_bounds__(LT *NSEG + 32 + 32 * NLB, MINB)
    quat_segwalk_bwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap dmap,
                            const float4 *__restrict__ carries, typename IO::elem *__restrict__ d_q,
                            typename IO::elem *__restrict__ d_init, unsigned int *__restrict__ ctr,
                            float4 *__restrict__ aggV, float4 *__restrict__ aggA, float4 *__restrict__ incl,
                            float4 *__restrict__ aggV_next, float4 *__restrict__ aggA_next,
                            float4 *__restrict__ incl_next, const Geometry geo, const Control ctl) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr int NT = LT * NSEG;   // compute threads
    constexpr int NW = NT / 32;     // compute warps
    static_assert(NT % 32 == 0 && LT <= 32, "compute threads are whole warps; one look-back thread per lane");
    constexpr uint32_t BQ = T * LT * IO::bytes;   // one operand of one chunk
    constexpr int TAB = K * NSEG * LT;            // entries of one unit's table
    constexpr int NSL = DL + 1;     // unit slots of the tables and of agg_ready / carry_ready
    constexpr int NU = 16;          // ticket slots (the producer is at most NST items = NST units ahead)
    static_assert(DL >= 1 && DL <= 3, "walk 2 lags walk 1 by one to three units");
    static_assert(NST + DL + 2 <= NU, "ticket slots: unit k - DL's is still held when unit k + NST's is written");
    static_assert(NST <= 3, "walk 1 of unit k + NSL ends at least 3 items after that of unit k");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    // Per unit (slot k % NSL), entry (chunk j, segment, lane): walk 1 writes the
    // segment's product into tab_a and its weighted sum into tab_w; the
    // look-back warp replaces them by the cum just before the segment (tab_a)
    // and the H entering it from the right (tab_w), which walk 2 reads.  An
    // entry is written and read by the same compute thread.
    float4 *tab_a = reinterpret_cast<float4 *>(ring + NST * 2 * BQ);
    float4 *tab_w = tab_a + NSL * TAB;
    __shared__ __align__(8) uint64_t full[NST], empty[NST];
    __shared__ __align__(8) uint64_t agg_ready[NSL], carry_ready[NSL];
    __shared__ int issued[NST];
    __shared__ int s_broken;
    __shared__ int s_unit[NU];      // producer -> compute: ticket of the CTA's k-th unit (slot k % NU), -1: end
    __shared__ int s_lbu[NSL];      // compute -> look-back: ticket of unit k (slot k % NSL), -1: end
    // Look-back warp: the carries entering unit k's chunks, copied into shared
    // memory while the look-back runs (K > 2), or held in registers.
    constexpr bool kFsmem = K > 2;
    __shared__ __align__(16) float4 s_F[kFsmem ? NSL : 1][kFsmem ? K : 1][LT];

    const int tid = static_cast<int>(threadIdx.x);
    const int NG = geo.NG, C = geo.C;
    const int P = (C + K - 1) / K;
    const int U = P * NG;

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
            issued[s] = 0;
        }
        for (int s = 0; s < NSL; ++s) {
            mbar_init(&agg_ready[s], NW);
            mbar_init(&carry_ready[s], 1);
        }
        for (int u = 0; u < NU; ++u) s_unit[u] = -1;
        fence_mbar_init();
        s_broken = 0;
    }
    __syncthreads();

    if (tid >= NT + 32) {
        // ======================= look-back warp(s) ============================
        static_assert(NLB == 1 || NLB == 2, "one look-back warp, or one per unit slot");
        const int wl = (tid - (NT + 32)) % 32;   // lane of the warp; lanes [0, LT) own the lane group's lanes
        const int lbw = (tid - (NT + 32)) / 32;  // which look-back warp: units k = lbw, lbw + NLB, ...
        const int lane = wl % LT;
        const bool own = wl < LT;
        for (int k = lbw;; k += NLB) {
            const int sl = k % NSL;
            if (!ws_wait(&agg_ready[sl], (k / NSL) & 1, ctl, -1, &s_broken)) break;
            const int t = s_lbu[sl];
            if (t < 0) break;
            const int p = t / NG, g = t - p * NG;
            const int b = g / geo.NGb;
            const int hj = (g - b * geo.NGb) * LT + lane;
            const int c_hi = C - p * K, c_lo = max(0, c_hi - K), n = c_hi - c_lo;
            if (own) {
                float4 *ta = tab_a + sl * TAB + lane, *tw = tab_w + sl * TAB + lane;
                float4 *sF = &s_F[kFsmem ? sl : 0][0][lane];
                float4 F[kFsmem ? 1 : K];
                // The carries entering the unit's chunks, fetched while the look-back runs.
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const bool real = j < n && hj < geo.HJ;
                    const float4 *src = carries + (static_cast<long long>(b) * C + c_lo + j) * geo.HJ + hj;
                    if constexpr (kFsmem) {
                        if (real) cp_async16(sF + j * LT, src);
                        else sF[j * LT] = q_ident();
                    } else {
                        F[j] = real ? __ldg(src) : q_ident();
                    }
                }
                // The unit's map: V = sum of conj(A_before) (x) w over its
                // segments in order, A their product.
                float4 V = q_zero(), A = q_ident();
                for (int e = 0; e < n * NSEG; e += NSEG) {
                    float4 av[NSEG], wv[NSEG];
#pragma unroll
                    for (int s = 0; s < NSEG; ++s) {
                        av[s] = ta[(e + s) * LT];
                        wv[s] = tw[(e + s) * LT];
                    }
#pragma unroll
                    for (int s = 0; s < NSEG; ++s) {
                        V = q_fma_cl(V, A, wv[s]);
                        A = q_mul(av[s], A);
                    }
                }
                const long long me = static_cast<long long>(t) * LT + lane;
                float4 H = q_zero();   // nothing enters the rightmost segment
                if (p > 0) {
                    __stcg(aggV + me, V);   // the map first: segments to the left can use it now
                    __stcg(aggA + me, A);
                    H = lookback_maps<LB>(aggV, aggA, incl, p, g, NG, LT, lane, ctl, c_lo * NG + g);
                }
                const float4 I = q_fma_cl(V, A, H);   // H at the unit's first step
                __stcg(incl + me, I);
                if (p == P - 1 && hj < geo.HJ) d_init[static_cast<long long>(b) * geo.HJ + hj] = IO::put(I);
                __stcg(aggV_next + me, lb_unpublished());   // this unit's entries of the next launch's buffers
                __stcg(aggA_next + me, lb_unpublished());
                __stcg(incl_next + me, lb_unpublished());
                // H entering each segment from the right, right to left, in place of w.
                for (int e = (n - 1) * NSEG; e >= 0; e -= NSEG) {
                    float4 av[NSEG], wv[NSEG];
#pragma unroll
                    for (int s = 0; s < NSEG; ++s) {
                        av[s] = ta[(e + s) * LT];
                        wv[s] = tw[(e + s) * LT];
                    }
#pragma unroll
                    for (int s = NSEG - 1; s >= 0; --s) {
                        tw[(e + s) * LT] = H;
                        H = q_fma_cl(wv[s], av[s], H);
                    }
                }
                // cum just before each segment, from its chunk's carry, in
                // place of the product; the K chains are independent.
                if constexpr (kFsmem) cp_async_wait_all();
                float4 X[K];
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if constexpr (kFsmem) X[j] = sF[j * LT];
                    else X[j] = F[j];
                }
#pragma unroll
                for (int s = 0; s < NSEG; ++s) {
#pragma unroll
                    for (int j = 0; j < K; ++j) {
                        if (j < n) {
                            const float4 a = ta[(j * NSEG + s) * LT];
                            ta[(j * NSEG + s) * LT] = X[j];
                            X[j] = q_mul(a, X[j]);
                        }
                    }
                }
            }
            __syncwarp();
            if (wl == 0) {
                mbar_arrive(&carry_ready[sl]);
                atomicAdd(ctr + 2, 1u);   // units done
            }
        }
    } else if (tid >= NT) {
        // ======================= producer warp ================================
        if (tid == NT) {
            const uint64_t keep = l2_policy_evict_last();
            const uint64_t drop = l2_policy_evict_first();
            int it = 0;   // items issued
            // Claim the stage of item `it` (its previous use released).
            auto claim = [&](int item) {
                const int st = it % NST;
                return it < NST || ws_wait(&empty[st], ((it / NST) - 1) & 1, ctl, item, &s_broken);
            };
            // Walk 1 takes the unit's chunks left to right, walk 2 in the
            // order W2FWD gives.
            auto walk = [&](int t, bool first) {
                const int p = t / NG, g = t - p * NG;
                const int b = g / geo.NGb, x0 = (g - b * geo.NGb) * LT * 4;
                const int c_hi = C - p * K, c_lo = max(0, c_hi - K), n = c_hi - c_lo;
                for (int j = 0; j < n; ++j) {
                    const int c = (first || W2FWD) ? c_lo + j : c_hi - 1 - j;
                    if (!claim(c * NG + g)) return false;
                    const int st = it % NST;
                    unsigned char *dst = ring + st * 2 * BQ;
                    ++issued[st];
                    mbar_arrive_expect_tx(&full[st], 2 * BQ + (first && c * NG + g == ctl.stall_tile ? 16u : 0u));
                    tma_load_3d_hint(dst, &qmap, x0, c * T, b, &full[st], first ? keep : drop);
                    tma_load_3d_hint(dst + BQ, &dmap, x0, c * T, b, &full[st], first ? keep : drop);
                    ++it;
                }
                return true;
            };
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int t = ld_volatile_int(&s_broken) ? U : static_cast<int>(atomicAdd(ctr, 1u));
                if (t >= U) {   // end marker where unit k's first load would be, then the pending second walks
                    if (claim(-1)) {
                        s_unit[k % NU] = -1;
                        mbar_arrive(&full[it % NST]);
                        ++it;
                        for (int j = max(0, k - DL); j < k && walk(s_unit[j % NU], false); ++j) {
                        }
                    }
                    break;
                }
                s_unit[k % NU] = t;   // read by the compute warps after the wait on this unit's first load
                ok = walk(t, true) && (k < DL || walk(s_unit[(k - DL) % NU], false));
            }
            if (ld_volatile_int(&s_broken)) {   // the loads issued get a bounded time to land
                for (int st = 0; st < NST; ++st) {
                    if (issued[st] == 0) continue;
                    const uint32_t parity = static_cast<uint32_t>(issued[st] - 1) & 1u;
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait(&full[st], parity) && global_timer_ns() - t0 <= ctl.timeout_ns) {
                    }
                }
            }
        }
    } else {
        // ======================= compute warps ================================
        // No block barrier: each warp walks the items in order on its own,
        // handing stages back through `empty` and units to the look-back warp
        // through `agg_ready` (one arrival per warp).
        const int lane = tid % LT, seg = tid / LT;
        const int cell0 = seg * N * LT + lane;
        const bool lead = (tid & 31) == 0;
        int it = 0;   // items consumed
        auto release = [&]() {   // this warp is done reading the stage of item `it`
            __syncwarp();
            if (lead) mbar_arrive(&empty[it % NST]);
            ++it;
        };
        // Walk 1 of unit t: every thread's segment product and weighted sum
        // into the unit's table (slot), then hand the unit on.
        auto walk1 = [&](int t, int slot) {
            const int p = t / NG, g = t - p * NG;
            const int c_hi = C - p * K, c_lo = max(0, c_hi - K), n = c_hi - c_lo;
            float4 *ta = tab_a + slot * TAB + seg * LT + lane, *tw = tab_w + slot * TAB + seg * LT + lane;
            for (int j = 0; j < n; ++j) {
                const int st = it % NST;
                ws_wait(&full[st], (it / NST) & 1, ctl, (c_lo + j) * NG + g, &s_broken);
                const E *Qt = reinterpret_cast<const E *>(ring + st * 2 * BQ);
                const E *Dt = Qt + T * LT;
                float4 loc = q_ident(), W = q_zero();
#pragma unroll
                for (int kk = 0; kk < N; ++kk) {
                    loc = q_mul(IO::get(Qt[cell0 + kk * LT]), loc);
                    W = q_fma_cl(W, loc, IO::get(Dt[cell0 + kk * LT]));
                }
                if (j + 1 < n) release();
                ta[j * NSEG * LT] = loc;
                tw[j * NSEG * LT] = W;
            }
            __syncwarp();
            if (lead) {
                if (tid == 0) s_lbu[slot] = t;
                mbar_arrive(&agg_ready[slot]);
            }
            // The last stage is handed back only after the unit: the producer
            // then refills it only once every warp has arrived for this unit,
            // which keeps the warps within one phase of agg_ready (each unit
            // is followed by at least NST items before the next unit of the
            // same slot ends).
            release();
        };
        // Walk 2 of unit t (slot): d_q, from the cum before and the H after
        // each segment in the table.
        auto walk2 = [&](int t, int slot) {
            const int p = t / NG, g = t - p * NG;
            const int b = g / geo.NGb;
            const int hj = (g - b * geo.NGb) * LT + lane;
            const bool lane_ok = hj < geo.HJ;
            const int c_hi = C - p * K, c_lo = max(0, c_hi - K), n = c_hi - c_lo;
            const long long row0 = static_cast<long long>(b) * geo.S;
            const float4 *ta = tab_a + slot * TAB + seg * LT + lane, *tw = tab_w + slot * TAB + seg * LT + lane;
            for (int jj = 0; jj < n; ++jj) {
                const int j = W2FWD ? jj : n - 1 - jj;
                const int c = c_lo + j;
                const int st = it % NST;
                ws_wait(&full[st], (it / NST) & 1, ctl, c * NG + g, &s_broken);
                const E *Qt = reinterpret_cast<const E *>(ring + st * 2 * BQ);
                const E *Dt = Qt + T * LT;
                float4 qv[N], dv[N], cp[N];
#pragma unroll
                for (int kk = 0; kk < N; ++kk) {
                    qv[kk] = IO::get(Qt[cell0 + kk * LT]);
                    dv[kk] = IO::get(Dt[cell0 + kk * LT]);
                }
                release();
                float4 X = ta[j * NSEG * LT];    // cum just before this segment
                float4 Hn = tw[j * NSEG * LT];   // H entering this segment from the right
#pragma unroll
                for (int kk = 0; kk < N; ++kk) {
                    cp[kk] = X;   // cum[t-1]
                    X = q_mul(qv[kk], X);
                }
                const long long t0 = static_cast<long long>(c) * T + seg * N;
                E *dst = d_q + (row0 + t0) * geo.HJ + hj;
                if (lane_ok && t0 + N <= geo.S) {
#pragma unroll
                    for (int kk = N - 1; kk >= 0; --kk) {
                        const float4 G = q_add(dv[kk], Hn);
                        __stcs(dst + static_cast<long long>(kk) * geo.HJ, IO::put(q_mul_cr(G, cp[kk])));
                        Hn = q_mul_cl(qv[kk], G);
                    }
                } else if (lane_ok) {
#pragma unroll
                    for (int kk = N - 1; kk >= 0; --kk) {
                        const float4 G = q_add(dv[kk], Hn);
                        if (t0 + kk < geo.S)
                            __stcs(dst + static_cast<long long>(kk) * geo.HJ, IO::put(q_mul_cr(G, cp[kk])));
                        Hn = q_mul_cl(qv[kk], G);
                    }
                }
            }
        };
        // Walk 2 of unit j, once its look-back is done.
        auto second = [&](int j) {
            ws_wait(&carry_ready[j % NSL], (j / NSL) & 1, ctl, -1, &s_broken);
            walk2(ld_volatile_int(&s_unit[j % NU]), j % NSL);
        };
        for (int k = 0;; ++k) {
            // Unit k: its first load (or the end marker) carries its ticket.
            const bool got = ws_wait(&full[it % NST], (it / NST) & 1, ctl, -1, &s_broken);
            const int t = got ? ld_volatile_int(&s_unit[k % NU]) : -1;
            if (t < 0) {
                if (got) release();   // the end marker's stage
                for (int j = max(0, k - DL); j < k; ++j) second(j);
                __syncwarp();
                if (lead) {   // the look-back warp(s) end too (every unit is done: the slots are free)
                    if (tid == 0) s_lbu[k % NSL] = -1;
                    mbar_arrive(&agg_ready[k % NSL]);
                    if (NLB == 2) {
                        if (tid == 0) s_lbu[(k + 1) % NSL] = -1;
                        mbar_arrive(&agg_ready[(k + 1) % NSL]);
                    }
                }
                break;
            }
            walk1(t, k % NSL);
            if (k >= DL) second(k - DL);
        }
    }
    __syncthreads();
    // The last CTA to finish resets the counters for the next launch, and the
    // next launch's buffers if units were left undone.
    __shared__ int s_last, s_short;
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(ctr + 1, 1u) == gridDim.x - 1;
        s_short = s_last && atomicAdd(ctr + 2, 0u) != static_cast<unsigned int>(U);
    }
    __syncthreads();
    if (s_last) {
        if (s_short) {
            const long long n = static_cast<long long>(U) * LT;
            for (long long i = tid; i < n; i += static_cast<long long>(blockDim.x)) {
                __stcg(aggV_next + i, lb_unpublished());
                __stcg(aggA_next + i, lb_unpublished());
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

// ---------------------------------------------------------------------------
// Carries-only pass: the forward carries of every chunk, carries[b, c] =
// cum[b, c*T - 1] (init for c = 0), from one read of q (16 bytes per
// element).  Units (segment p of K chunks from the left, lane group g),
// u = p * NG + g, as in the forward segmented walk; there is one walk per
// unit.  The compute warps write the product of each thread's N steps of each
// chunk into the unit's table and walk on, with no block barrier; the
// look-back warp folds the table into the unit's product A (noting the
// product before each chunk), publishes it, looks back for the carry X
// entering the unit, publishes A (x) X and writes the unit's carries.  The
// look-back values and tickets work as in quat_segwalk_bwd_kernel.
// ---------------------------------------------------------------------------
template <typename IO, int LT, int NSEG, int N, int NST, int K, int LB = 4, int NLB = 1>
__global__ void __launch_bounds__(LT *NSEG + 32 + 32 * NLB)
    quat_carries_pass_kernel(const __grid_constant__ CUtensorMap qmap, const typename IO::elem *__restrict__ init,
                             float4 *__restrict__ carries, unsigned int *__restrict__ ctr, float4 *__restrict__ agg,
                             float4 *__restrict__ incl, float4 *__restrict__ agg_next, float4 *__restrict__ incl_next,
                             const Geometry geo, const Control ctl) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr int NT = LT * NSEG;
    constexpr int NW = NT / 32;
    static_assert(NT % 32 == 0 && LT <= 32, "compute threads are whole warps; one look-back thread per lane");
    constexpr uint32_t BYTES = T * LT * IO::bytes;
    constexpr int TAB = K * NSEG * LT;
    constexpr int NU = 16;
    static_assert(NST + 3 <= NU, "unit slots");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    float4 *tab_a = reinterpret_cast<float4 *>(ring + NST * BYTES);   // [2][K][NSEG][LT]: products of N steps
    __shared__ __align__(8) uint64_t full[NST], empty[NST];
    __shared__ __align__(8) uint64_t agg_ready[2], carry_ready[2];
    __shared__ int issued[NST];
    __shared__ int s_broken;
    __shared__ int s_unit[NU];
    __shared__ int s_lbu[2];

    const int tid = static_cast<int>(threadIdx.x);
    const int NG = geo.NG, C = geo.C;
    const int P = (C + K - 1) / K;
    const int U = P * NG;

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
            issued[s] = 0;
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&agg_ready[s], NW);
            mbar_init(&carry_ready[s], 1);
        }
        for (int u = 0; u < NU; ++u) s_unit[u] = -1;
        fence_mbar_init();
        s_broken = 0;
    }
    __syncthreads();

    if (tid >= NT + 32) {
        // ======================= look-back warp(s) ============================
        static_assert(NLB == 1 || NLB == 2, "one look-back warp, or one per unit slot");
        const int wl = (tid - (NT + 32)) % 32;
        const int lbw = (tid - (NT + 32)) / 32;   // units k = lbw, lbw + NLB, ...
        const int lane = wl % LT;
        const bool own = wl < LT;
        for (int k = lbw;; k += NLB) {
            if (!ws_wait(&agg_ready[k & 1], (k >> 1) & 1, ctl, -1, &s_broken)) break;
            const int t = s_lbu[k & 1];
            if (t < 0) break;
            const int p = t / NG, g = t - p * NG;
            const int b = g / geo.NGb;
            const int hj = (g - b * geo.NGb) * LT + lane;
            const bool lane_ok = hj < geo.HJ;
            const int c0 = p * K, n = min(K, C - c0);
            const float4 *ta = tab_a + (k & 1) * TAB + lane;
            float4 Ab[K];   // the unit's product before each chunk
            float4 A = q_ident();
            float4 X = q_ident();
            if (own) {
                if (p == 0 && lane_ok) X = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    Ab[j] = A;
                    if (j < n) {
                        float4 av[NSEG];
#pragma unroll
                        for (int s = 0; s < NSEG; ++s) av[s] = ta[(j * NSEG + s) * LT];
#pragma unroll
                        for (int s = 0; s < NSEG; ++s) A = q_mul(av[s], A);
                    }
                }
            }
            const long long me = static_cast<long long>(t) * LT + lane;
            if (p > 0) {
                if (own) __stcg(agg + me, A);   // the product first: later segments can use it now
                if (own) X = lookback_products<LB>(agg, incl, p, g, NG, LT, lane, ctl, c0 * NG + g);
            }
            if (own) {
                __stcg(incl + me, q_mul(A, X));
                __stcg(agg_next + me, lb_unpublished());   // this unit's entries of the next launch's buffers
                __stcg(incl_next + me, lb_unpublished());
                if (lane_ok) {
                    float4 *dst = carries + (static_cast<long long>(b) * C + c0) * geo.HJ + hj;
#pragma unroll
                    for (int j = 0; j < K; ++j)
                        if (j < n) dst[static_cast<long long>(j) * geo.HJ] = q_mul(Ab[j], X);
                }
            }
            __syncwarp();
            if (wl == 0) {
                mbar_arrive(&carry_ready[k & 1]);
                atomicAdd(ctr + 2, 1u);   // units done
            }
        }
    } else if (tid >= NT) {
        // ======================= producer warp ================================
        if (tid == NT) {
            int it = 0;   // items issued
            auto claim = [&](int item) {
                const int st = it % NST;
                return it < NST || ws_wait(&empty[st], ((it / NST) - 1) & 1, ctl, item, &s_broken);
            };
            for (int k = 0;; ++k) {
                const int t = ld_volatile_int(&s_broken) ? U : static_cast<int>(atomicAdd(ctr, 1u));
                if (t >= U) {   // end marker where unit k's first load would be
                    if (claim(-1)) {
                        s_unit[k % NU] = -1;
                        mbar_arrive(&full[it % NST]);
                        ++it;
                    }
                    break;
                }
                s_unit[k % NU] = t;
                const int p = t / NG, g = t - p * NG;
                const int b = g / geo.NGb, x0 = (g - b * geo.NGb) * LT * 4;
                const int c0 = p * K, n = min(K, C - c0);
                bool ok = true;
                for (int j = 0; j < n && ok; ++j) {
                    const int c = c0 + j;
                    ok = claim(c * NG + g);
                    if (!ok) break;
                    const int st = it % NST;
                    ++issued[st];
                    mbar_arrive_expect_tx(&full[st], BYTES + (c * NG + g == ctl.stall_tile ? 16u : 0u));
                    tma_load_3d(ring + st * BYTES, &qmap, x0, c * T, b, &full[st]);
                    ++it;
                }
                if (!ok) break;
            }
            if (ld_volatile_int(&s_broken)) {   // the loads issued get a bounded time to land
                for (int st = 0; st < NST; ++st) {
                    if (issued[st] == 0) continue;
                    const uint32_t parity = static_cast<uint32_t>(issued[st] - 1) & 1u;
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait(&full[st], parity) && global_timer_ns() - t0 <= ctl.timeout_ns) {
                    }
                }
            }
        }
    } else {
        // ======================= compute warps ================================
        const int lane = tid % LT, seg = tid / LT;
        const int cell0 = seg * N * LT + lane;
        const bool lead = (tid & 31) == 0;
        int it = 0;
        auto release = [&]() {
            __syncwarp();
            if (lead) mbar_arrive(&empty[it % NST]);
            ++it;
        };
        for (int k = 0;; ++k) {
            // Slot k & 1 (and s_lbu[k & 1]) are free once the look-back warp is
            // done with unit k - 2.
            if (k >= 2) ws_wait(&carry_ready[k & 1], ((k - 2) >> 1) & 1, ctl, -1, &s_broken);
            const bool got = ws_wait(&full[it % NST], (it / NST) & 1, ctl, -1, &s_broken);
            const int t = got ? ld_volatile_int(&s_unit[k % NU]) : -1;
            __syncwarp();
            if (t < 0) {
                if (got) release();   // the end marker's stage
                // (two look-back warps: the other slot is free once unit k - 1 is done)
                if (NLB == 2 && k >= 1) ws_wait(&carry_ready[(k - 1) & 1], ((k - 1) >> 1) & 1, ctl, -1, &s_broken);
                __syncwarp();
                if (lead) {   // the look-back warp(s) end too
                    if (tid == 0) s_lbu[k & 1] = -1;
                    mbar_arrive(&agg_ready[k & 1]);
                    if (NLB == 2) {
                        if (tid == 0) s_lbu[(k + 1) & 1] = -1;
                        mbar_arrive(&agg_ready[(k + 1) & 1]);
                    }
                }
                break;
            }
            const int p = t / NG, g = t - p * NG;
            const int c0 = p * K, n = min(K, C - c0);
            float4 *ta = tab_a + (k & 1) * TAB + seg * LT + lane;
            for (int j = 0; j < n; ++j) {
                const int st = it % NST;
                ws_wait(&full[st], (it / NST) & 1, ctl, (c0 + j) * NG + g, &s_broken);
                const E *Qt = reinterpret_cast<const E *>(ring + st * BYTES);
                float4 loc = q_ident();
#pragma unroll
                for (int kk = 0; kk < N; ++kk) loc = q_mul(IO::get(Qt[cell0 + kk * LT]), loc);
                if (j + 1 < n) release();
                ta[j * NSEG * LT] = loc;
            }
            __syncwarp();
            if (lead) {
                if (tid == 0) s_lbu[k & 1] = t;
                mbar_arrive(&agg_ready[k & 1]);
            }
            release();
        }
    }
    __syncthreads();
    __shared__ int s_last, s_short;
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(ctr + 1, 1u) == gridDim.x - 1;
        s_short = s_last && atomicAdd(ctr + 2, 0u) != static_cast<unsigned int>(U);
    }
    __syncthreads();
    if (s_last) {
        if (s_short) {
            const long long n = static_cast<long long>(U) * LT;
            for (long long i = tid; i < n; i += static_cast<long long>(blockDim.x)) {
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

// Dynamic shared memory of the carries pass: the ring, then the two unit
// slots of the table.
__host__ __device__ constexpr size_t carries_pass_smem_bytes(int lt, int nseg, int n, int nst, int k, int eb = 16) {
    return 128 + size_t(nst) * nseg * n * lt * eb + size_t(2) * k * nseg * lt * 16;
}

// Dynamic shared memory: the ring (two operands per stage), then the nsl
// unit slots of the two tables (nsl = DL + 1).
__host__ __device__ constexpr size_t segwalk_bwd_smem_bytes(int lt, int nseg, int n, int nst, int k, int eb = 16,
                                                            int nsl = 2) {
    return 128 + size_t(nst) * 2 * nseg * n * lt * eb + size_t(2) * nsl * k * nseg * lt * 16;
}

}  // namespace qs
