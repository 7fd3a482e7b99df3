// quat_segwalk_ws.cuh -- the segmented chained walk (forward) in
// warp-specialised CTAs: compute warps, a producer warp and a look-back warp.
#pragma once

#include "quat_segwalk.cuh"

namespace qs {

// ---------------------------------------------------------------------------
// The same units, walks and look-back as quat_segwalk_fwd_kernel, with the
// work of a CTA split by warp:
//
//   * compute warps (LT * NSEG threads) walk in the order
//       W1(u0), W1(u1), W2(u0), W1(u2), W2(u1), ...
//     (W1: first walk, the segment product; W2: second walk, cum), so a
//     unit's look-back runs while the next unit's first walk does.  They
//     synchronise among themselves on named barrier 1.
//   * the producer warp (one thread) takes the tickets and issues every TMA
//     load in that item order through one NST-stage ring.  A stage is refilled
//     once every compute warp has released it (full / empty mbarriers), so the
//     producer waits on no compute barrier.  When no unit is left it posts an
//     end marker (a zero-byte arrival) where the next unit's first load would
//     be, then the last second walk.
//   * the look-back warp (one thread per lane) takes a unit's segment product
//     from the compute warps, publishes it, folds the earlier segments into
//     the carry, publishes the inclusive value and hands the carry back.  It
//     writes nothing else, so its release stores do not wait behind the cum
//     stream.
//
// Every wait is bounded; after one runs out the CTA stops taking units,
// waits no more and ends.  Units it took but did not publish make later
// look-backs run out their own limit (bounded) and publish NaN.
// ---------------------------------------------------------------------------

// Bounded wait on an mbarrier phase: false if it ran out (recorded, `broken`
// set) or the CTA is already broken.
__device__ __forceinline__ bool ws_wait(uint64_t *bar, uint32_t parity, const Control &ctl, int item, int *broken) {
    if (ld_volatile_int(broken)) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (ld_volatile_int(broken)) return false;
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            record_error(ctl.hdr, item);
            *reinterpret_cast<volatile int *>(broken) = 1;
            return false;
        }
    }
    return true;
}

template <int NT>
__device__ __forceinline__ void compute_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// Look-back of one lane (decoupled look-back over the segments of its lane
// group).  A round loads the LB nearest predecessors not yet folded, together
// (one memory latency), and folds the published ones in order, up to the
// first inclusive value; at the first one not yet published it stops and the
// next round loads afresh from there, so a value loaded before a wait is
// never used after it.  Only the nearest unfolded predecessor is waited for.
// A predecessor counts as published once none of its words holds the
// all-ones pattern.  A wait that runs out is recorded (as `item`) and gives NaN.

// H entering segment p of lane group g from the right: the maps of segments
// p-1, p-2, ... composed back to the nearest published inclusive value.
template <int LB>
__device__ __forceinline__ float4 lookback_maps(const float4 *aggV, const float4 *aggA, const float4 *incl, int p,
                                                int g, int NG, int LT, int lane, const Control &ctl, int item) {
    // H_right = aV + aM (x) (what lies further right)
    float4 aV = q_zero(), aM = q_ident();
    int base = p - 1;
    for (;;) {
        float4 v[LB], a[LB], h[LB];
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            const long long idx = (static_cast<long long>(base - j < 0 ? 0 : base - j) * NG + g) * LT + lane;
            h[j] = __ldcg(incl + idx);
            v[j] = __ldcg(aggV + idx);
            a[j] = __ldcg(aggA + idx);
        }
        int folded = 0;
        bool gap = false;
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            if (gap) continue;
            if (base - j < 0) return aV;   // past the right end of the sequence: H = 0 there
            if (lb_published(h[j])) return q_fma(aV, aM, h[j]);
            if (lb_published(v[j]) && lb_published(a[j])) {
                aV = q_fma(aV, aM, v[j]);
                aM = q_mul_cr(aM, a[j]);
                ++folded;
            } else {
                gap = true;
            }
        }
        base -= folded;
        if (folded > 0) continue;
        // The nearest predecessor is not published yet: wait for it.
        const long long idx = (static_cast<long long>(base) * NG + g) * LT + lane;
        const unsigned long long t0 = global_timer_ns();
        float4 hv, vv, av;
        do {
            if (global_timer_ns() - t0 > ctl.timeout_ns) {
                record_error(ctl.hdr, item);
                return q_nan();
            }
            hv = __ldcg(incl + idx);
            vv = __ldcg(aggV + idx);
            av = __ldcg(aggA + idx);
        } while (!lb_published(hv) && !(lb_published(vv) && lb_published(av)));
        if (lb_published(hv)) return q_fma(aV, aM, hv);
        aV = q_fma(aV, aM, vv);
        aM = q_mul_cr(aM, av);
        --base;
    }
}

// The carry entering segment p of lane group g from the left (forward): the
// products of segments p-1, p-2, ... back to the nearest published inclusive
// value, the product itself included.
template <int LB>
__device__ __forceinline__ float4 lookback_products(const float4 *agg, const float4 *incl, int p, int g, int NG,
                                                    int LT, int lane, const Control &ctl, int item) {
    float4 acc = q_ident();
    int base = p - 1;
    for (;;) {
        float4 av[LB], iv[LB];
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            const long long idx = (static_cast<long long>(base - j < 0 ? 0 : base - j) * NG + g) * LT + lane;
            av[j] = __ldcg(agg + idx);
            iv[j] = __ldcg(incl + idx);
        }
        int folded = 0;
        bool gap = false;
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            if (gap) continue;
            if (base - j < 0) return acc;   // before segment 0: an inclusive identity
            if (lb_published(iv[j])) return q_mul(acc, iv[j]);
            if (lb_published(av[j])) {
                acc = q_mul(acc, av[j]);
                ++folded;
            } else {
                gap = true;
            }
        }
        base -= folded;
        if (folded > 0) continue;
        const long long idx = (static_cast<long long>(base) * NG + g) * LT + lane;
        const unsigned long long t0 = global_timer_ns();
        float4 a1, i1;
        do {
            if (global_timer_ns() - t0 > ctl.timeout_ns) {
                record_error(ctl.hdr, item);
                return q_nan();
            }
            a1 = __ldcg(agg + idx);
            i1 = __ldcg(incl + idx);
        } while (!lb_published(i1) && !lb_published(a1));
        if (lb_published(i1)) return q_mul(acc, i1);
        acc = q_mul(acc, a1);
        --base;
    }
}

// The carry entering segment p of lane group g for one lane, from look-back
// values that carry their own state (see quat_segwalk_fwd_kernel, SENT): per
// round the LB predecessors' products and inclusive values are loaded
// together, one memory latency.  NaN if a wait ran out (recorded as `item`).
template <int LB>
__device__ __forceinline__ float4 segment_lookback_values(const float4 *agg, const float4 *incl, int p, int g, int NG,
                                                          int LT, int lane, const Control &ctl, int item) {
    float4 acc = q_ident();
    for (int base = p - 1;; base -= LB) {
        float4 av[LB], iv[LB];
        long long idx[LB];
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            const int pp = base - j;
            idx[j] = (static_cast<long long>(pp < 0 ? 0 : pp) * NG + g) * LT + lane;
            av[j] = q_ident();
            iv[j] = q_ident();
            if (pp >= 0) {
                av[j] = __ldcg(agg + idx[j]);
                iv[j] = __ldcg(incl + idx[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < LB; ++j) {
            if (base - j < 0) return acc;   // before segment 0: an inclusive identity
            if (!lb_published(iv[j]) && !lb_published(av[j])) {
                const unsigned long long t0 = global_timer_ns();
                do {
                    if (global_timer_ns() - t0 > ctl.timeout_ns) {
                        record_error(ctl.hdr, item);
                        return q_nan();
                    }
                    av[j] = __ldcg(agg + idx[j]);
                    iv[j] = __ldcg(incl + idx[j]);
                } while (!lb_published(iv[j]) && !lb_published(av[j]));
            }
            if (lb_published(iv[j])) return q_mul(acc, iv[j]);
            acc = q_mul(acc, av[j]);
        }
    }
}

// `carries` (may be null): [B, C, H*J] float4, the state entering every
// chunk, carries[b, c] = cum[b, c*T - 1] (init for c = 0).
template <typename IO, int LT, int NSEG, int N, int NST, int K, bool SENT = false>
__global__ void __launch_bounds__(LT *NSEG + 64)
    quat_segwalk_ws_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const typename IO::elem *__restrict__ init,
                               typename IO::elem *__restrict__ out, float4 *__restrict__ carries,
                               uint32_t *__restrict__ flags, unsigned int *__restrict__ ctr,
                               float4 *__restrict__ agg, float4 *__restrict__ incl, float4 *__restrict__ agg_next,
                               float4 *__restrict__ incl_next, const Geometry geo, const Control ctl,
                               uint32_t epoch) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr int NT = LT * NSEG;   // compute threads
    constexpr int NW = NT / 32;     // compute warps
    static_assert(NT % 32 == 0 && LT <= 32, "compute threads are whole warps; one look-back thread per lane");
    constexpr uint32_t BYTES = T * LT * IO::bytes;
    constexpr int NU = 16;          // unit slots (the producer is at most NST items = NST units ahead)
    static_assert(NST + 3 <= NU, "unit slots");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    __shared__ __align__(8) uint64_t full[NST], empty[NST];
    __shared__ __align__(8) uint64_t agg_ready[2], carry_ready[2];
    __shared__ int issued[NST];
    __shared__ int s_broken;
    __shared__ int s_unit[NU];      // producer -> compute: ticket of the CTA's k-th unit (slot k % NU), -1: end
    __shared__ int s_cur;           // compute thread 0 -> compute warps: the current unit's ticket
    __shared__ int s_lbu[2];        // compute -> look-back: ticket of unit k (slot k & 1), -1: end
    __shared__ float4 s_a[2][NSEG][LT];   // segment products of an item (slot: item parity)
    __shared__ float4 s_x[2][LT];         // carry into an item of a second walk (slot: item parity)
    __shared__ float4 s_A[2][LT];         // segment product of unit k (slot k & 1)
    __shared__ float4 s_X[2][LT];         // carry into unit k (slot k & 1)

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
            mbar_init(&agg_ready[s], 1);
            mbar_init(&carry_ready[s], 1);
        }
        for (int u = 0; u < NU; ++u) s_unit[u] = -1;
        fence_mbar_init();
        s_broken = 0;
    }
    __syncthreads();

    if (tid >= NT + 32) {
        // ======================= look-back warp ===============================
        const int lane = tid - (NT + 32);
        const uint32_t tag = epoch << 2;
        for (int k = 0;; ++k) {
            if (!ws_wait(&agg_ready[k & 1], (k >> 1) & 1, ctl, -1, &s_broken)) break;
            const int t = s_lbu[k & 1];
            if (t < 0) break;
            const int p = t / NG, g = t - p * NG;
            const int b = g / geo.NGb;
            const int hj = (g - b * geo.NGb) * LT + lane;
            if (lane < LT) {
                const float4 A = s_A[k & 1][lane];
                const long long me = static_cast<long long>(t) * LT + lane;
                float4 acc = q_ident();
                if (p == 0) {
                    if (hj < geo.HJ) acc = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
                } else if constexpr (SENT) {
                    __stcg(agg + me, A);   // the product first: later segments can use it now
                    acc = segment_lookback_values<8>(agg, incl, p, g, NG, LT, lane, ctl, p * K * NG + g);
                } else {
                    __stcg(agg + me, A);   // the product first: later segments can use it now
                    st_release_u32(flags + me, tag | CH_AGG);
                    // acc = A_{p-1} (x) A_{p-2} (x) ... (x) incl: LB predecessors per
                    // round, their status words loaded together, then their values.
                    constexpr int LB = 8;
                    bool done = false;
                    for (int base = p - 1; !done; base -= LB) {
                        uint32_t f[LB];
                        long long idx[LB];
#pragma unroll
                        for (int j = 0; j < LB; ++j) {
                            const int pp = base - j;   // before segment 0: an inclusive identity
                            idx[j] = (static_cast<long long>(pp < 0 ? 0 : pp) * NG + g) * LT + lane;
                            f[j] = pp < 0 ? (tag | CH_INCL) : ld_acquire_u32(flags + idx[j]);
                        }
                        bool lost = false;
#pragma unroll
                        for (int j = 0; j < LB; ++j) {
                            if (lost || (f[j] & ~3u) == tag) continue;
                            const unsigned long long t0 = global_timer_ns();
                            do {
                                if (global_timer_ns() - t0 > ctl.timeout_ns) {
                                    record_error(ctl.hdr, p * K * NG + g);
                                    lost = true;
                                    break;
                                }
                                f[j] = ld_acquire_u32(flags + idx[j]);
                            } while ((f[j] & ~3u) != tag);
                        }
                        if (lost) {
                            acc = q_nan();
                            break;
                        }
                        float4 v[LB];
                        bool stop = false;
#pragma unroll
                        for (int j = 0; j < LB; ++j) {   // the values to fold, loaded together
                            const bool inc = (f[j] & 3u) == CH_INCL;
                            v[j] = q_ident();
                            if (!stop && base - j >= 0) v[j] = inc ? __ldcg(incl + idx[j]) : __ldcg(agg + idx[j]);
                            stop = stop || inc;
                        }
#pragma unroll
                        for (int j = 0; j < LB; ++j) {
                            if (done) break;
                            acc = q_mul(acc, v[j]);
                            done = (f[j] & 3u) == CH_INCL;
                        }
                    }
                }
                __stcg(incl + me, q_mul(A, acc));
                if constexpr (SENT) {   // this unit's entries of the next launch's buffers
                    __stcg(agg_next + me, lb_unpublished());
                    __stcg(incl_next + me, lb_unpublished());
                } else {
                    st_release_u32(flags + me, tag | CH_INCL);
                }
                s_X[k & 1][lane] = acc;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&carry_ready[k & 1]);
                if constexpr (SENT) atomicAdd(ctr + 2, 1u);   // units done
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
                s_unit[k % NU] = t;   // read by compute thread 0 after the wait on this unit's first load
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
        int it = 0;   // items consumed
        auto release = [&]() {   // this warp is done reading the stage of item `it`
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(&empty[it % NST]);
            ++it;
        };
        // First walk of unit t: the segment product into s_A[slot], then
        // hand the unit to the look-back warp.
        auto walk1 = [&](int t, int slot) {
            const int p = t / NG, g = t - p * NG;
            const int c0 = p * K, n = min(K, C - c0);
            float4 A = q_ident();   // segment-0 threads
            for (int j = 0; j < n; ++j) {
                const int st = it % NST, sl = it & 1;
                ws_wait(&full[st], (it / NST) & 1, ctl, (c0 + j) * NG + g, &s_broken);
                const E *Qt = reinterpret_cast<const E *>(ring + st * BYTES);
                float4 loc = q_ident();
#pragma unroll
                for (int kk = 0; kk < N; ++kk) loc = q_mul(IO::get(Qt[(seg * N + kk) * LT + lane]), loc);
                release();
                s_a[sl][seg][lane] = loc;
                compute_sync<NT>();
                if (seg == 0) {
#pragma unroll
                    for (int kk = 0; kk < NSEG; ++kk) A = q_mul(s_a[sl][kk][lane], A);
                }
            }
            if (seg == 0) s_A[slot][lane] = A;
            compute_sync<NT>();
            if (tid == 0) {
                s_lbu[slot] = t;
                mbar_arrive(&agg_ready[slot]);
            }
        };
        // Second walk of unit t from the carry X: cum.
        auto walk2 = [&](int t, float4 X) {
            const int p = t / NG, g = t - p * NG;
            const int b = g / geo.NGb;
            const int hj = (g - b * geo.NGb) * LT + lane;
            const bool lane_ok = hj < geo.HJ;
            const int c0 = p * K, n = min(K, C - c0);
            const long long row0 = static_cast<long long>(b) * geo.S;
            float4 R = X;   // segment-0 threads: carry into the next chunk
            if (seg == 0) s_x[it & 1][lane] = X;
            compute_sync<NT>();
            for (int j = 0; j < n; ++j) {
                const int st = it % NST, sl = it & 1;
                ws_wait(&full[st], (it / NST) & 1, ctl, (c0 + j) * NG + g, &s_broken);
                const E *Qt = reinterpret_cast<const E *>(ring + st * BYTES);
                float4 x[N];
                float4 loc = q_ident();
#pragma unroll
                for (int kk = 0; kk < N; ++kk) {
                    loc = q_mul(IO::get(Qt[(seg * N + kk) * LT + lane]), loc);
                    x[kk] = loc;
                }
                release();
                s_a[sl][seg][lane] = loc;
                compute_sync<NT>();
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
                        if (t0 + kk < geo.S)
                            __stcs(dst + static_cast<long long>(kk) * geo.HJ, IO::put(q_mul(x[kk], Y)));
                }
            }
        };
        int prev = -1;
        for (int k = 0;; ++k) {
            // Unit k: its first load (or the end marker) carries its ticket.
            if (tid == 0) {
                const bool got = ws_wait(&full[it % NST], (it / NST) & 1, ctl, -1, &s_broken);
                s_cur = got ? ld_volatile_int(&s_unit[k % NU]) : -1;
            }
            compute_sync<NT>();
            const int t = s_cur;
            compute_sync<NT>();   // s_cur is read before it is written again
            if (t < 0) {
                release();        // the end marker's stage
                if (prev >= 0) {
                    ws_wait(&carry_ready[(k - 1) & 1], ((k - 1) >> 1) & 1, ctl, -1, &s_broken);
                    walk2(prev, s_X[(k - 1) & 1][lane]);
                }
                if (tid == 0) {   // the look-back warp ends too
                    s_lbu[k & 1] = -1;
                    mbar_arrive(&agg_ready[k & 1]);
                }
                break;
            }
            walk1(t, k & 1);
            if (prev >= 0) {
                ws_wait(&carry_ready[(k - 1) & 1], ((k - 1) >> 1) & 1, ctl, -1, &s_broken);
                walk2(prev, s_X[(k - 1) & 1][lane]);
            }
            prev = t;
        }
    }
    __syncthreads();
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

}  // namespace qs
