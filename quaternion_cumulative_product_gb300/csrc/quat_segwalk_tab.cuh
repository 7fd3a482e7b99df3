// quat_segwalk_tab.cuh -- the segmented chained walk of the forward without
// block barriers: per-unit tables in shared memory carry what the serial
// folds of a unit produce, and the folds run on look-back warps.
#pragma once

#include "quat_segwalk_ws.cuh"

namespace qs {

// ---------------------------------------------------------------------------
// Units, tickets, look-back values and item order as in
// quat_segwalk_ws_fwd_kernel (unit u = p * NG + g is segment p of K chunks,
// counted from the left, of lane group g; items W1(u0) W1(u1) W2(u0) W1(u2)
// W2(u1) ...), with the work of a unit split this way:
//
//   1. walk 1 (q loaded evict-last): every compute thread writes the product
//      of its N steps of each chunk into the unit's table, and walks on;
//   2. a look-back warp folds the table in order into the unit's product A,
//      noting in each entry the product of the unit before it, publishes A,
//      looks back for the carry X entering the unit, publishes A (x) X, and
//      replaces every entry by the cum just before that thread's steps (the
//      entry (x) X); with `carries`, it also writes the carry entering every
//      chunk;
//   3. walk 2 (from L2, evict-first): every thread walks its N steps from its
//      table entry, cum[t] = q_t (x) cum[t-1].
//
// One quaternion product per element in each walk, no block barrier: the
// compute warps hand stages back through `empty` and units on through
// `agg_ready` (one arrival per warp after its last table write), and wait for
// the look-back result of a unit (`carry_ready`) only before its second walk.
// With NLB = 2 look-back warps unit k goes to warp k % 2.  Every wait is
// bounded; after one runs out the CTA stops taking units and ends, and units
// it took but did not publish make later look-backs run out (NaN).
// ---------------------------------------------------------------------------
template <typename IO, int LT, int NSEG, int N, int NST, int K, int NLB = 1, int LB = 4>
__global__ void __launch_bounds__(LT *NSEG + 32 + 32 * NLB)
    quat_segwalk_tab_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const typename IO::elem *__restrict__ init,
                                typename IO::elem *__restrict__ out, float4 *__restrict__ carries,
                                unsigned int *__restrict__ ctr, float4 *__restrict__ agg, float4 *__restrict__ incl,
                                float4 *__restrict__ agg_next, float4 *__restrict__ incl_next, const Geometry geo,
                                const Control ctl) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr int NT = LT * NSEG;   // compute threads
    constexpr int NW = NT / 32;     // compute warps
    static_assert(NT % 32 == 0 && LT <= 32, "compute threads are whole warps; one look-back thread per lane");
    static_assert(NLB == 1 || NLB == 2, "one look-back warp, or one per unit slot");
    static_assert(NST <= 3, "walk 1 of unit k + 2 ends at least 3 items after that of unit k");
    constexpr uint32_t BYTES = T * LT * IO::bytes;
    constexpr int TAB = K * NSEG * LT;   // entries of one unit's table
    constexpr int NU = 16;
    static_assert(NST + 3 <= NU, "unit slots");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    float4 *tab = reinterpret_cast<float4 *>(ring + NST * BYTES);   // [2][K][NSEG][LT]
    __shared__ __align__(8) uint64_t full[NST], empty[NST];
    __shared__ __align__(8) uint64_t agg_ready[2], carry_ready[2];
    __shared__ int issued[NST];
    __shared__ int s_broken;
    __shared__ int s_unit[NU];   // producer -> compute: ticket of the CTA's k-th unit (slot k % NU), -1: end
    __shared__ int s_lbu[2];     // compute -> look-back: ticket of unit k (slot k & 1), -1: end

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
            if (own) {
                float4 *ta = tab + (k & 1) * TAB + lane;
                // The unit's product, each entry replaced by the product before it.
                float4 A = q_ident();
                for (int e = 0; e < n * NSEG; e += NSEG) {
                    float4 av[NSEG];
#pragma unroll
                    for (int s = 0; s < NSEG; ++s) av[s] = ta[(e + s) * LT];
#pragma unroll
                    for (int s = 0; s < NSEG; ++s) {
                        ta[(e + s) * LT] = A;
                        A = q_mul(av[s], A);
                    }
                }
                const long long me = static_cast<long long>(t) * LT + lane;
                float4 X = q_ident();
                if (p == 0) {
                    if (lane_ok) X = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
                } else {
                    __stcg(agg + me, A);   // the product first: later segments can use it now
                    X = lookback_products<LB>(agg, incl, p, g, NG, LT, lane, ctl, c0 * NG + g);
                }
                __stcg(incl + me, q_mul(A, X));
                __stcg(agg_next + me, lb_unpublished());   // this unit's entries of the next launch's buffers
                __stcg(incl_next + me, lb_unpublished());
                // cum just before every thread's steps; the carry entering each chunk.
                float4 *car = (carries != nullptr && lane_ok)
                                  ? carries + (static_cast<long long>(b) * C + c0) * geo.HJ + hj
                                  : nullptr;
                for (int e = 0; e < n * NSEG; e += NSEG) {
#pragma unroll
                    for (int s = 0; s < NSEG; ++s) {
                        const float4 x = q_mul(ta[(e + s) * LT], X);
                        ta[(e + s) * LT] = x;
                        if (s == 0 && car != nullptr) car[static_cast<long long>(e / NSEG) * geo.HJ] = x;
                    }
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
            const uint64_t keep = l2_policy_evict_last();
            const uint64_t drop = l2_policy_evict_first();
            int it = 0;   // items issued
            auto claim = [&](int item) {
                const int st = it % NST;
                return it < NST || ws_wait(&empty[st], ((it / NST) - 1) & 1, ctl, item, &s_broken);
            };
            // Both walks take the unit's chunks left to right.
            auto walk = [&](int t, bool first) {
                const int p = t / NG, g = t - p * NG;
                const int b = g / geo.NGb, x0 = (g - b * geo.NGb) * LT * 4;
                const int c0 = p * K, n = min(K, C - c0);
                for (int j = 0; j < n; ++j) {
                    const int c = c0 + j;
                    if (!claim(c * NG + g)) return false;
                    const int st = it % NST;
                    ++issued[st];
                    mbar_arrive_expect_tx(&full[st], BYTES + (first && c * NG + g == ctl.stall_tile ? 16u : 0u));
                    tma_load_3d_hint(ring + st * BYTES, &qmap, x0, c * T, b, &full[st], first ? keep : drop);
                    ++it;
                }
                return true;
            };
            int prev = -1;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int t = ld_volatile_int(&s_broken) ? U : static_cast<int>(atomicAdd(ctr, 1u));
                if (t >= U) {   // end marker where unit k's first load would be
                    if (claim(-1)) {
                        s_unit[k % NU] = -1;
                        mbar_arrive(&full[it % NST]);
                        ++it;
                        if (prev >= 0) walk(prev, false);
                    }
                    break;
                }
                s_unit[k % NU] = t;
                ok = walk(t, true) && (prev < 0 || walk(prev, false));
                prev = t;
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
        int it = 0;   // items consumed
        auto release = [&]() {
            __syncwarp();
            if (lead) mbar_arrive(&empty[it % NST]);
            ++it;
        };
        auto walk1 = [&](int t, int slot) {
            const int p = t / NG, g = t - p * NG;
            const int c0 = p * K, n = min(K, C - c0);
            float4 *ta = tab + slot * TAB + seg * LT + lane;
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
                if (tid == 0) s_lbu[slot] = t;
                mbar_arrive(&agg_ready[slot]);
            }
            release();   // the last stage only after the unit is handed on (see quat_segwalk_bwd_kernel)
        };
        auto walk2 = [&](int t, int slot) {
            const int p = t / NG, g = t - p * NG;
            const int b = g / geo.NGb;
            const int hj = (g - b * geo.NGb) * LT + lane;
            const bool lane_ok = hj < geo.HJ;
            const int c0 = p * K, n = min(K, C - c0);
            const long long row0 = static_cast<long long>(b) * geo.S;
            const float4 *ta = tab + slot * TAB + seg * LT + lane;
            for (int j = 0; j < n; ++j) {
                const int st = it % NST;
                ws_wait(&full[st], (it / NST) & 1, ctl, (c0 + j) * NG + g, &s_broken);
                const E *Qt = reinterpret_cast<const E *>(ring + st * BYTES);
                float4 qv[N];
#pragma unroll
                for (int kk = 0; kk < N; ++kk) qv[kk] = IO::get(Qt[cell0 + kk * LT]);
                release();
                float4 X = ta[j * NSEG * LT];   // cum just before this thread's steps
                const long long t0 = static_cast<long long>(c0 + j) * T + seg * N;
                E *dst = out + (row0 + t0) * geo.HJ + hj;
                if (lane_ok && t0 + N <= geo.S) {
#pragma unroll
                    for (int kk = 0; kk < N; ++kk) {
                        X = q_mul(qv[kk], X);
                        __stcs(dst + static_cast<long long>(kk) * geo.HJ, IO::put(X));
                    }
                } else if (lane_ok) {
#pragma unroll
                    for (int kk = 0; kk < N; ++kk) {
                        X = q_mul(qv[kk], X);
                        if (t0 + kk < geo.S) __stcs(dst + static_cast<long long>(kk) * geo.HJ, IO::put(X));
                    }
                }
            }
        };
        int prev = -1;
        for (int k = 0;; ++k) {
            const bool got = ws_wait(&full[it % NST], (it / NST) & 1, ctl, -1, &s_broken);
            const int t = got ? ld_volatile_int(&s_unit[k % NU]) : -1;
            if (t < 0) {
                if (got) release();   // the end marker's stage
                if (prev >= 0) {
                    ws_wait(&carry_ready[(k - 1) & 1], ((k - 1) >> 1) & 1, ctl, -1, &s_broken);
                    walk2(prev, (k - 1) & 1);
                }
                __syncwarp();
                if (lead) {   // the look-back warp(s) end too (unit k - 1 is done: its slot is free)
                    if (tid == 0) s_lbu[k & 1] = -1;
                    mbar_arrive(&agg_ready[k & 1]);
                    if (NLB == 2) {
                        if (tid == 0) s_lbu[(k + 1) & 1] = -1;
                        mbar_arrive(&agg_ready[(k + 1) & 1]);
                    }
                }
                break;
            }
            walk1(t, k & 1);
            if (prev >= 0) {
                ws_wait(&carry_ready[(k - 1) & 1], ((k - 1) >> 1) & 1, ctl, -1, &s_broken);
                walk2(prev, (k - 1) & 1);
            }
            prev = t;
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

// Dynamic shared memory: the ring, then the two unit slots of the table.
__host__ __device__ constexpr size_t segwalk_tab_smem_bytes(int lt, int nseg, int n, int nst, int k, int eb = 16) {
    return 128 + size_t(nst) * nseg * n * lt * eb + size_t(2) * k * nseg * lt * 16;
}

}  // namespace qs
