// quat_walk.cuh -- the walk kernels (one CTA per lane group walks the whole
// sequence) and their shared-memory sizes.
#pragma once

#include "quat_common.cuh"

namespace qs {

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
    __shared__ int issued[NST];   // loads issued per stage (by the producer thread)
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
    // The loads are issued by the first thread of the first warp without
    // segment-0 threads (segment 0 carries the lane after the barrier; the
    // low segments have the fewest products to fold): a stall on a full TMA
    // queue then delays no thread on the chunk's critical path.
    constexpr int kWarp1 = (LT + 31) / 32 * 32;
    const bool producer = threadIdx.x == (kWarp1 < LT * NSEG ? kWarp1 : LT * NSEG - 1);
    if (producer)
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
        if (producer && !s_broken && c + NST < C) issue(c + NST);
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
//
// A CTA walks lane groups blockIdx.x, blockIdx.x + gridDim.x, ... one after
// the other (both walks of one group before the next group), so the grid
// sets how many groups are in flight at once; the rings and shared slots
// carry over from one group to the next.
// MINB: CTAs per SM the register allocation must allow (ptxas caps the
// registers per thread accordingly).
template <typename IO, int LT, int NSEG, int N, int NSTF, int NSTB, bool SELF, bool GIVEN, int MINB = 1>
__global__ void __launch_bounds__(LT *NSEG, MINB)
    quat_walk_bwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap dmap,
                         const typename IO::elem *__restrict__ init, float4 *__restrict__ carF,
                         const float4 *__restrict__ given, typename IO::elem *__restrict__ d_q,
                         typename IO::elem *__restrict__ d_init, const Geometry geo, const Control ctl) {
    using E = typename IO::elem;
    constexpr int T = NSEG * N;
    constexpr uint32_t BQ = T * LT * IO::bytes;   // one operand of one chunk
    extern __shared__ unsigned char smem_raw[];
    unsigned char *ring = align128(smem_raw);
    const int tid = static_cast<int>(threadIdx.x);
    __shared__ __align__(8) uint64_t fullF[NSTF];
    __shared__ __align__(8) uint64_t fullB[NSTB];
    __shared__ int issuedF[NSTF], issuedB[NSTB];
    __shared__ int s_broken;
    __shared__ float4 s_a[2][NSEG][LT];             // segment products (slot: chunk parity)
    __shared__ float4 s_w[SELF ? 2 : 1][NSEG][LT];  // segment weighted sums (reverse walk)
    __shared__ float4 s_x[SELF ? 1 : NSEG][LT];     // cum just before each segment
    __shared__ float4 s_h[SELF ? 2 : NSEG][LT];     // H entering each segment / the next chunk

    const int lane = tid % LT, seg = tid / LT;
    const int C = geo.C;
    const long long NL = geo.NL;

    if (tid == 0) {
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

    // Ring items (chunks) of the groups this CTA walked before the current
    // one: stage = item % ring depth, phase parity = (item / depth) & 1.
    int baseF = 0, baseB = 0;
    const bool producer = tid == LT * NSEG - 1;   // issues every load (it never folds)
    for (int g = static_cast<int>(blockIdx.x); g < geo.NG; g += static_cast<int>(gridDim.x)) {
        const int b = g / geo.NGb, x0 = (g - b * geo.NGb) * LT * 4;
        const int hj = (g - b * geo.NGb) * LT + lane;
        const bool lane_ok = hj < geo.HJ;
        const long long col = static_cast<long long>(g) * LT + lane;   // padded lane of this thread

        if constexpr (!GIVEN) {
            // ---- forward walk over q: carries F_c ----------------------------
            const uint64_t keep = l2_policy_evict_last();
            auto issueF = [&](int c) {
                const int st = (baseF + c) % NSTF;
                ++issuedF[st];
                mbar_arrive_expect_tx(&fullF[st], BQ + (c * geo.NG + g == ctl.stall_tile ? 16u : 0u));
                tma_load_3d_hint(ring + st * BQ, &qmap, x0, c * T, b, &fullF[st], keep);
            };
            if (producer && !s_broken)
                for (int c = 0; c < NSTF && c < C; ++c) issueF(c);

            float4 R = q_ident();
            if (seg == 0 && lane_ok) R = IO::get(init[static_cast<long long>(b) * geo.HJ + hj]);
            for (int c = 0; c < C; ++c) {
                const int it = baseF + c, st = it % NSTF, sl = c & 1;
                const E *Qt = reinterpret_cast<const E *>(ring + st * BQ);
                if (!ld_volatile_int(&s_broken) && !wait_stage(&fullF[st], (it / NSTF) & 1, ctl, c * geo.NG + g))
                    s_broken = 1;
                float4 loc = q_ident();
#pragma unroll
                for (int k = 0; k < N; ++k) loc = q_mul(IO::get(Qt[(seg * N + k) * LT + lane]), loc);
                s_a[sl][seg][lane] = loc;
                __syncthreads();
                if (producer && !s_broken && c + NSTF < C) issueF(c + NSTF);
                if (seg == 0) {   // segment 0 carries the lane through the chunk
                    carF[static_cast<long long>(c) * NL + col] = R;
#pragma unroll
                    for (int k = 0; k < NSEG; ++k) R = q_mul(s_a[sl][k][lane], R);
                }
            }
            baseF += C;
        }
        __syncthreads();   // every read of the forward ring is done before the reverse ring reuses it

        // ---- reverse walk over q and d_cum: d_q, d_init ----------------------
        auto issueB = [&](int j) {   // reverse step j covers chunk C-1-j
            const int st = (baseB + j) % NSTB, c = C - 1 - j;
            ++issuedB[st];
            unsigned char *dst = ring + st * 2 * BQ;
            mbar_arrive_expect_tx(&fullB[st], 2 * BQ);
            tma_load_3d_hint(dst, &qmap, x0, c * T, b, &fullB[st], drop);
            tma_load_3d_hint(dst + BQ, &dmap, x0, c * T, b, &fullB[st], drop);
        };
        if (producer && !s_broken)
            for (int j = 0; j < NSTB && j < C; ++j) issueB(j);

        float4 Hc = q_zero();   // H entering the current chunk from the right (segment-1 threads; every thread if SELF)
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
            const int it = baseB + j, st = it % NSTB, sl = j & 1;
            const float4 F = F_next;
            if ((SELF || seg == 0) && c > 0) F_next = carry_of(c - 1);
            const E *Qt = reinterpret_cast<const E *>(ring + st * 2 * BQ);
            const E *Dt = Qt + T * LT;
            if (!ld_volatile_int(&s_broken) && !wait_stage(&fullB[st], (it / NSTB) & 1, ctl, c * geo.NG + g))
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
            if (producer && !s_broken && j + NSTB < C) issueB(j + NSTB);
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
                if (seg < 2) {
                    // Two chains of NSEG steps y <- Q + A (x) y: the carry
                    // forward through the segments on the segment-0 threads
                    // (A = s_a[k], Q = 0) and H backward through them on the
                    // segment-1 threads (A = conj(s_a[k]), Q = s_w[k], k
                    // descending).  Written as one instruction stream, so the
                    // two segments run side by side when they share a warp.
                    const bool back = seg == 1;
                    const float sg = back ? -1.f : 1.f;
                    float4(*out)[LT] = back ? s_h : s_x;
                    float4 y = back ? Hc : F;
                    const int step = back ? -1 : 1;
                    // Every step's operands are loaded before the chain starts, so
                    // no shared-memory latency sits between two of its steps.
                    float4 Ak[NSEG], Qk[NSEG];
                    int idx = back ? NSEG - 1 : 0;
#pragma unroll
                    for (int k = 0; k < NSEG; ++k, idx += step) {
                        float4 A = s_a[sl][idx][lane];
                        const float4 Wk = s_w[0][idx][lane];
                        A.y *= sg;
                        A.z *= sg;
                        A.w *= sg;
                        Ak[k] = A;
                        Qk[k] = make_float4(back ? Wk.x : 0.f, back ? Wk.y : 0.f, back ? Wk.z : 0.f, back ? Wk.w : 0.f);
                    }
                    idx = back ? NSEG - 1 : 0;
#pragma unroll
                    for (int k = 0; k < NSEG; ++k, idx += step) {
                        out[idx][lane] = y;
                        y = q_fma(Qk[k], Ak[k], y);
                    }
                    if (back) {
                        Hc = y;
                        if (c == 0 && lane_ok) d_init[static_cast<long long>(b) * geo.HJ + hj] = IO::put(Hc);
                    }
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
                    if (t0 + k < geo.S)
                        __stcs(dst + static_cast<long long>(k) * geo.HJ, IO::put(q_mul_cr(G, q_mul(lp[k], X))));
                    Hn = q_mul_cl(qv[k], G);
                }
            }
        }
        baseB += C;
        // Every read of this group's ring stages and shared slots is done
        // before the next group's loads and writes reuse them.
        __syncthreads();
    }
    if (s_broken) {
        drain_ring<NSTF>(fullF, issuedF, ctl);
        drain_ring<NSTB>(fullB, issuedB, ctl);
    }
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
