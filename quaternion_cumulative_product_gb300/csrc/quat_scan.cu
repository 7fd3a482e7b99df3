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
//  * A tile is LT = 32 lanes x T consecutive steps.  Its rows (one step, 32
//    lanes = 512 contiguous bytes) are staged into shared memory by one 3-D TMA
//    load per operand, double/triple buffered in a persistent CTA that claims
//    tiles from a global counter.  Inside the tile, thread (seg, lane) owns N
//    consecutive steps of one lane; 8 segments per tile.
//
//  * Forward: per-thread sequential products give the segment-local prefixes,
//    warp 0 scans the 8 segment aggregates, and a decoupled look-back over the
//    tiles of the same lane group (earlier chunks) gives the carry cum[t0-1].
//    Tile aggregate = L_c = local product of the chunk; inclusive value =
//    cum at the chunk's last step.  Output cum[t] = local_t (x) carry.
//
//  * Backward: the page's per-chunk aggregates are the chunk product L_c and the
//    weighted sum W_c = sum_{s in c} conj(local_s) (x) d_cum[s].  Writing
//    H[t] = conj(q_t) (x) G[t] (the cotangent that step t hands to cum[t-1]),
//    a chunk maps the H entering at its end to the H at its start by the affine
//    map  H_c = W_c + conj(L_c) (x) H_{c+1}.  This is exactly the page's
//    factorisation conj(P_s) = conj(P_{c-1}) (x) conj(local_s) of the suffix
//    sum, and it is exact for all quaternions (no unit assumption), because it
//    composes the literal reverse recurrence.  d_init = H_0.
//    d_q needs both directions: the forward carry cum[t0-1] (from earlier
//    chunks) and H_{c+1} (from later chunks).  One persistent kernel runs two
//    kinds of work items from one queue: "A" items (read q only, forward
//    look-back, publish cum at each chunk end) and "C" items (read q and d_cum,
//    reverse look-back over the affine aggregates, wait for the A carry of the
//    previous chunk, write d_q).  Lanes are processed in batches small enough
//    that a batch's q stays in L2 between its A pass and its C pass; the queue
//    runs A(0), A(1), C(0), A(2), C(1), ...  Every wait is on an item claimed
//    earlier from the queue, so the schedule cannot deadlock; every wait is also
//    bounded in time and reports QS_ERR_TIMEOUT instead of hanging.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "quat_cumprod.h"
#include "quat_device.cuh"

namespace qs {

constexpr int LT = 32;                 // lanes per tile (= warp width)
constexpr int NTHREADS = 256;          // threads per CTA
constexpr int NSEG = NTHREADS / LT;    // sequence segments per tile
constexpr uint32_t ST_AGG = 1;         // flag: tile aggregate published
constexpr uint32_t ST_INCL = 2;        // flag: inclusive carry published

// Per-workspace control block (device memory, zero-initialised, epoch = 1).
struct __align__(256) WsHeader {
    unsigned int counter;     // next work item
    unsigned int done;        // CTAs that finished the current launch
    unsigned int epoch;       // tag of the current launch's flags
    unsigned int err_epoch;   // epoch of the last launch that gave up waiting
    unsigned int err_code;    // 1 once a wait ran out (cleared by quat_cumprod_status)
    unsigned int err_count;   // number of waits that ran out
    unsigned long long err_item;  // first work item that ran out
};

struct Geometry {
    long long S;   // sequence length
    int HJ;        // lanes per batch entry (H*J)
    int NGb;       // lane groups per batch entry
    int NG;        // lane groups in total
    int C;         // chunks along the sequence
    int boxw;      // lanes per TMA box row (min(LT, HJ))
    int boxh;      // rows per TMA box (min(T, S))
};

struct Control {
    WsHeader *hdr;
    int nitems;
    int stall_item;
    unsigned long long timeout_ns;
};

struct BwdArrays {
    unsigned long long *a_flags;  // [CA*NG]
    float4 *a_agg;                // [CA*NG*LT]   chunk product L_c
    float4 *a_incl;               // [CA*NG*LT]   cum at the chunk's last step
    unsigned long long *c_flags;  // [C*NG]
    float4 *c_agg;                // [C*NG*LT*2]  affine map (conj(L_c), W_c)
    float4 *c_incl;               // [C*NG*LT]    H at the chunk's first step
};

struct Schedule {
    int CA;   // chunks with an A item (C - 1)
    int GB;   // lane groups per batch
    int NB;   // batches
};

__device__ __forceinline__ unsigned long long pack_flag(uint32_t epoch, uint32_t st) {
    return (static_cast<unsigned long long>(epoch) << 2) | st;
}

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ void record_error(WsHeader *h, uint32_t epoch, int item) {
    if (atomicCAS(&h->err_code, 0u, 1u) == 0u) h->err_item = static_cast<unsigned long long>(item);
    atomicAdd(&h->err_count, 1u);
    atomicExch(&h->err_epoch, epoch);
}

// Waits until `flag` carries this launch's epoch with a status >= need.
// Bounded: gives up after ctl.timeout_ns (records the error) or as soon as
// another CTA of this launch has given up; `failed` is then set.
__device__ __noinline__ uint32_t wait_flag(const unsigned long long *flag, uint32_t epoch,
                                           const Control &ctl, int item, uint32_t need, bool &failed) {
    unsigned long long f = ld_acquire_u64(flag);
    if (static_cast<uint32_t>(f >> 2) == epoch && static_cast<uint32_t>(f & 3u) >= need)
        return static_cast<uint32_t>(f & 3u);
    const unsigned long long t0 = global_timer_ns();
    unsigned ns = 32;
    for (;;) {
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
        f = ld_acquire_u64(flag);
        if (static_cast<uint32_t>(f >> 2) == epoch && static_cast<uint32_t>(f & 3u) >= need)
            return static_cast<uint32_t>(f & 3u);
        if (ld_volatile_u32(&ctl.hdr->err_epoch) == epoch) {
            failed = true;
            return ST_INCL;
        }
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            record_error(ctl.hdr, epoch, item);
            failed = true;
            return ST_INCL;
        }
    }
}

// Waits for a TMA stage; bounded like wait_flag (a TMA copy completes in
// microseconds, so running out here means the device is in trouble).
__device__ __forceinline__ void wait_stage(uint64_t *bar, uint32_t parity, const Control &ctl,
                                           uint32_t epoch, int item) {
    if (mbar_try_wait(bar, parity)) return;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            record_error(ctl.hdr, epoch, item);
            return;
        }
    }
}

// Warp 0 publishes one quaternion per lane, then the flag (release).
__device__ __forceinline__ void publish1(float4 *vals, unsigned long long *flag, long long idx, int lane,
                                         float4 v, unsigned long long fv) {
    __stcg(vals + idx * LT + lane, v);
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_u64(flag, fv);
}

__device__ __forceinline__ void publish2(float4 *vals, unsigned long long *flag, long long idx, int lane,
                                         float4 m, float4 v, unsigned long long fv) {
    __stcg(vals + (idx * LT + lane) * 2, m);
    __stcg(vals + (idx * LT + lane) * 2 + 1, v);
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_u64(flag, fv);
}

// Decoupled look-back in the forward direction.  Tile (chunk, g) needs the
// exclusive carry cum[t0-1] = L_{chunk-1} (x) ... (x) L_0 (x) init, combined
// from the nearest tiles before it: each published aggregate (L) or inclusive
// value (cum at that tile's end, which ends the walk).  Segment `seg` of the
// block reads predecessor chunk-1-seg, so one round looks NSEG tiles back.
// All threads call it; the result is valid in threads with seg == 0.
__device__ float4 lookback_prod(const unsigned long long *flags, const float4 *agg, const float4 *incl,
                                int chunk, int g, int NG, float4 init_v, uint32_t epoch, const Control &ctl,
                                int item, int seg, int lane, float4 (*s_lb)[LT], uint32_t *s_st, int *s_done) {
    float4 acc = q_ident();
    int base = chunk - 1;
    for (;;) {
        const int pc = base - seg;
        float4 v;
        uint32_t st;
        if (pc < 0) {
            st = ST_INCL;   // before the first chunk: cum[-1] = init
            v = init_v;
        } else {
            const long long pidx = static_cast<long long>(pc) * NG + g;
            bool failed = false;
            st = wait_flag(flags + pidx, epoch, ctl, item, ST_AGG, failed);
            if (failed)
                v = q_nan();
            else
                v = (st == ST_INCL) ? __ldcg(incl + pidx * LT + lane) : __ldcg(agg + pidx * LT + lane);
        }
        s_lb[seg][lane] = v;
        if (lane == 0) s_st[seg] = st;
        __syncthreads();
        if (seg == 0) {
            int done = 0;
            for (int k = 0; k < NSEG; ++k) {
                acc = q_mul(acc, s_lb[k][lane]);
                if (s_st[k] == ST_INCL) {
                    done = 1;
                    break;
                }
            }
            if (lane == 0) *s_done = done;
        }
        __syncthreads();
        if (*s_done) break;
        base -= NSEG;
    }
    return acc;
}

// Decoupled look-back in the reverse direction over affine maps
// x -> V + M (x) x (M = conj(L_c), V = W_c for an aggregate; an inclusive value
// is H at that tile's first step and ends the walk).  Returns H_{chunk+1}, the
// cotangent entering tile `chunk` from the right; valid in threads seg == 0.
__device__ float4 lookback_affine(const unsigned long long *flags, const float4 *agg2, const float4 *incl,
                                  int chunk, int C, int g, int NG, uint32_t epoch, const Control &ctl, int item,
                                  int seg, int lane, float4 (*s_lb)[LT][2], uint32_t *s_st, int *s_done) {
    float4 accM = q_ident(), accV = q_zero();
    int base = chunk + 1;
    for (;;) {
        const int pc = base + seg;
        float4 m = q_zero(), v = q_zero();
        uint32_t st;
        if (pc >= C) {
            st = ST_INCL;   // past the last step: nothing flows back
        } else {
            const long long pidx = static_cast<long long>(pc) * NG + g;
            bool failed = false;
            st = wait_flag(flags + pidx, epoch, ctl, item, ST_AGG, failed);
            if (failed) {
                v = q_nan();
            } else if (st == ST_INCL) {
                v = __ldcg(incl + pidx * LT + lane);
            } else {
                m = __ldcg(agg2 + (pidx * LT + lane) * 2);
                v = __ldcg(agg2 + (pidx * LT + lane) * 2 + 1);
            }
        }
        s_lb[seg][lane][0] = m;
        s_lb[seg][lane][1] = v;
        if (lane == 0) s_st[seg] = st;
        __syncthreads();
        if (seg == 0) {
            int done = 0;
            for (int k = 0; k < NSEG; ++k) {
                accV = q_add(accV, q_mul(accM, s_lb[k][lane][1]));
                if (s_st[k] == ST_INCL) {
                    done = 1;
                    break;
                }
                accM = q_mul(accM, s_lb[k][lane][0]);
            }
            if (lane == 0) *s_done = done;
        }
        __syncthreads();
        if (*s_done) break;
        base += NSEG;
    }
    return accV;
}

// The last CTA to finish resets the queue and advances the epoch, so that the
// next launch on this workspace needs no memset.
__device__ __forceinline__ void finish_launch(const Control &ctl, uint32_t epoch) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&ctl.hdr->done, 1u);
        if (prev == gridDim.x - 1) {
            ctl.hdr->counter = 0;
            ctl.hdr->done = 0;
            __threadfence();
            ctl.hdr->epoch = (epoch + 1 == 0) ? 1 : epoch + 1;
        }
    }
}

// ---------------------------------------------------------------------------
// Backward work-item schedule: A(0), [A(1), C(0)], [A(2), C(1)], ..., C(NB-1).
// Within A(k) items are chunk-major in increasing chunk order; within C(k)
// chunk-major in decreasing chunk order.  Batch k holds lane groups
// [k*GB, k*GB + gk).
// ---------------------------------------------------------------------------
struct Work {
    int phase;   // 0 = A item, 1 = C item
    int chunk;
    int g;
};

__host__ __device__ inline Work decode_bwd(int id, int NG, int C, const Schedule &s) {
    const int last_g = NG - (s.NB - 1) * s.GB;
    const int fullA = s.CA * s.GB, fullC = C * s.GB;
    const int nA0 = s.CA * (s.NB == 1 ? last_g : s.GB);
    int phase, k, local;
    int r = id;
    if (r < nA0) {
        phase = 0;
        k = 0;
        local = r;
    } else {
        r -= nA0;
        const int nfull = s.NB > 2 ? s.NB - 2 : 0;   // pairs [A(k), C(k-1)] for k = 1..NB-2
        const long long pair = static_cast<long long>(fullA) + fullC;
        if (static_cast<long long>(r) < nfull * pair) {
            k = 1 + static_cast<int>(r / pair);
            r = static_cast<int>(r % pair);
            if (r < fullA) {
                phase = 0;
                local = r;
            } else {
                phase = 1;
                k -= 1;
                local = r - fullA;
            }
        } else {
            r -= static_cast<int>(nfull * pair);
            if (s.NB >= 2) {
                const int kk = s.NB - 1;
                const int nAk = s.CA * last_g;
                if (r < nAk) {
                    phase = 0;
                    k = kk;
                    local = r;
                } else if (r - nAk < fullC) {
                    phase = 1;
                    k = kk - 1;
                    local = r - nAk;
                } else {
                    phase = 1;
                    k = kk;
                    local = r - nAk - fullC;
                }
            } else {
                phase = 1;
                k = 0;
                local = r;
            }
        }
    }
    const int gk = (k == s.NB - 1) ? last_g : s.GB;
    Work w;
    w.phase = phase;
    w.g = k * s.GB + local % gk;
    w.chunk = (phase == 0) ? local / gk : C - 1 - local / gk;
    return w;
}

// ---------------------------------------------------------------------------
// Forward kernel.
// ---------------------------------------------------------------------------
template <int N, int NST>
__global__ void __launch_bounds__(NTHREADS)
    quat_scan_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const float4 *__restrict__ init,
                         float4 *__restrict__ cum, unsigned long long *flags, float4 *agg, float4 *incl,
                         const Geometry geo, const Control ctl) {
    static_assert(NST >= 2, "at least double buffering");
    constexpr int T = NSEG * N;
    constexpr uint32_t STAGE_BYTES = T * LT * 16;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar[NST];
    __shared__ int s_items[NST];
    __shared__ float4 s_seg[NSEG][LT];
    __shared__ float4 s_lb[NSEG][LT];
    __shared__ uint32_t s_st[NSEG];
    __shared__ float4 s_carry[LT];
    __shared__ int s_done;

    const int tid = threadIdx.x, lane = tid % LT, seg = tid / LT;
    const uint32_t epoch = ld_volatile_u32(&ctl.hdr->epoch);
    const uint32_t box_bytes = static_cast<uint32_t>(geo.boxw) * geo.boxh * 16u;
    const long long S = geo.S;
    const int HJ = geo.HJ, NG = geo.NG;

    auto issue = [&](int it, int stage) {
        const int chunk = it / NG, g = it % NG;
        const int b = g / geo.NGb, hj0 = (g % geo.NGb) * LT;
        mbar_arrive_expect_tx(&bar[stage], box_bytes);
        tma_load_3d(smem + stage * STAGE_BYTES, &qmap, hj0 * 4, chunk * T, b, &bar[stage]);
    };

    if (tid == 0) {
        prefetch_tensormap(&qmap);
        for (int s = 0; s < NST; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        for (int s = 0; s < NST - 1; ++s) {
            const int it = static_cast<int>(atomicAdd(&ctl.hdr->counter, 1u));
            s_items[s] = it;
            if (it < ctl.nitems) issue(it, s);
        }
    }
    __syncthreads();

    uint32_t phases = 0;
    int head = 0;
    for (;;) {
        const int item = s_items[head];
        if (item >= ctl.nitems) break;
        if (tid == 0) {
            const int nx = static_cast<int>(atomicAdd(&ctl.hdr->counter, 1u));
            const int st = (head + NST - 1) % NST;
            s_items[st] = nx;
            if (nx < ctl.nitems) {
                fence_proxy_async_smem();
                issue(nx, st);
            }
        }
        wait_stage(&bar[head], (phases >> head) & 1u, ctl, epoch, item);
        phases ^= 1u << head;

        const int chunk = item / NG, g = item % NG;
        const int b = g / geo.NGb, hj = (g % geo.NGb) * LT + lane;
        const bool lane_ok = lane < geo.boxw && hj < HJ;
        const float4 *tile = reinterpret_cast<const float4 *>(smem + head * STAGE_BYTES);
        const long long t0 = static_cast<long long>(chunk) * T + seg * N;

        // Segment-local prefix products: x[i] = q_{t0+i} (x) ... (x) q_{t0}.
        float4 x[N];
        float4 loc = q_ident();
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float4 v = tile[(seg * N + i) * geo.boxw + lane];
            if (t0 + i >= S) v = q_zero();
            loc = q_mul(v, loc);
            x[i] = loc;
        }
        s_seg[seg][lane] = loc;
        __syncthreads();

        float4 Lc = q_ident();
        if (seg == 0) {
            // Exclusive prefixes of the segment aggregates (in place), chunk product L_c.
            float4 e = q_ident();
#pragma unroll
            for (int k = 0; k < NSEG; ++k) {
                const float4 a = s_seg[k][lane];
                s_seg[k][lane] = e;
                e = q_mul(a, e);
            }
            Lc = e;
            if (chunk > 0 && item != ctl.stall_item)
                publish1(agg, flags + item, item, lane, Lc, pack_flag(epoch, ST_AGG));
        }
        const float4 init_v = lane_ok ? init[static_cast<long long>(b) * HJ + hj] : q_ident();
        float4 carry = init_v;
        if (chunk > 0)
            carry = lookback_prod(flags, agg, incl, chunk, g, NG, init_v, epoch, ctl, item, seg, lane, s_lb, s_st,
                                  &s_done);
        if (seg == 0) {
            if (item != ctl.stall_item)
                publish1(incl, flags + item, item, lane, q_mul(Lc, carry), pack_flag(epoch, ST_INCL));
            s_carry[lane] = carry;
        }
        __syncthreads();

        const float4 X = q_mul(s_seg[seg][lane], s_carry[lane]);   // cum just before this segment
        if (lane_ok) {
            float4 *out = cum + (static_cast<long long>(b) * S + t0) * HJ + hj;
#pragma unroll
            for (int i = 0; i < N; ++i)
                if (t0 + i < S) __stcs(out + static_cast<long long>(i) * HJ, q_mul(x[i], X));
        }
        __syncthreads();
        head = (head + 1) % NST;
    }
    finish_launch(ctl, epoch);
}

// ---------------------------------------------------------------------------
// Backward kernel (A and C items from one queue).
// ---------------------------------------------------------------------------
template <int N, int NST>
__global__ void __launch_bounds__(NTHREADS)
    quat_scan_bwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap dmap,
                         const float4 *__restrict__ init, float4 *__restrict__ d_q, float4 *__restrict__ d_init,
                         const BwdArrays arr, const Geometry geo, const Schedule sch, const Control ctl) {
    static_assert(NST >= 2, "at least double buffering");
    constexpr int T = NSEG * N;
    constexpr uint32_t HALF_BYTES = T * LT * 16;    // one operand of a stage
    constexpr uint32_t STAGE_BYTES = 2 * HALF_BYTES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar[NST];
    __shared__ int s_items[NST];
    __shared__ float4 s_seg[NSEG][LT];   // segment products, then exclusive prefixes
    __shared__ float4 s_w[NSEG][LT];     // segment weighted sums, then V of the suffix map
    __shared__ float4 s_m[NSEG][LT];     // M of the suffix map
    __shared__ float4 s_lb[NSEG][LT][2];
    __shared__ uint32_t s_st[NSEG];
    __shared__ float4 s_carry[LT];
    __shared__ float4 s_h[LT];
    __shared__ int s_done;

    const int tid = threadIdx.x, lane = tid % LT, seg = tid / LT;
    const uint32_t epoch = ld_volatile_u32(&ctl.hdr->epoch);
    const uint32_t box_bytes = static_cast<uint32_t>(geo.boxw) * geo.boxh * 16u;
    const long long S = geo.S;
    const int HJ = geo.HJ, NG = geo.NG, C = geo.C;

    auto issue = [&](int it, int stage) {
        const Work w = decode_bwd(it, NG, C, sch);
        const int b = w.g / geo.NGb, hj0 = (w.g % geo.NGb) * LT;
        unsigned char *dst = smem + stage * STAGE_BYTES;
        if (w.phase == 0) {
            mbar_arrive_expect_tx(&bar[stage], box_bytes);
            tma_load_3d(dst, &qmap, hj0 * 4, w.chunk * T, b, &bar[stage]);
        } else {
            mbar_arrive_expect_tx(&bar[stage], 2 * box_bytes);
            tma_load_3d(dst, &qmap, hj0 * 4, w.chunk * T, b, &bar[stage]);
            tma_load_3d(dst + HALF_BYTES, &dmap, hj0 * 4, w.chunk * T, b, &bar[stage]);
        }
    };

    if (tid == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&dmap);
        for (int s = 0; s < NST; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        for (int s = 0; s < NST - 1; ++s) {
            const int it = static_cast<int>(atomicAdd(&ctl.hdr->counter, 1u));
            s_items[s] = it;
            if (it < ctl.nitems) issue(it, s);
        }
    }
    __syncthreads();

    uint32_t phases = 0;
    int head = 0;
    for (;;) {
        const int item = s_items[head];
        if (item >= ctl.nitems) break;
        if (tid == 0) {
            const int nx = static_cast<int>(atomicAdd(&ctl.hdr->counter, 1u));
            const int st = (head + NST - 1) % NST;
            s_items[st] = nx;
            if (nx < ctl.nitems) {
                fence_proxy_async_smem();
                issue(nx, st);
            }
        }
        wait_stage(&bar[head], (phases >> head) & 1u, ctl, epoch, item);
        phases ^= 1u << head;

        const Work w = decode_bwd(item, NG, C, sch);
        const int chunk = w.chunk, g = w.g;
        const int b = g / geo.NGb, hj = (g % geo.NGb) * LT + lane;
        const bool lane_ok = lane < geo.boxw && hj < HJ;
        const long long idx = static_cast<long long>(chunk) * NG + g;
        const float4 *Qt = reinterpret_cast<const float4 *>(smem + head * STAGE_BYTES);
        const float4 *Dt = reinterpret_cast<const float4 *>(smem + head * STAGE_BYTES + HALF_BYTES);
        const long long t0 = static_cast<long long>(chunk) * T + seg * N;
        const float4 init_v = lane_ok ? init[static_cast<long long>(b) * HJ + hj] : q_ident();

        if (w.phase == 0) {
            // ---- A item: forward carry at the end of this chunk ----------------
            float4 loc = q_ident();
#pragma unroll
            for (int i = 0; i < N; ++i) {
                float4 v = Qt[(seg * N + i) * geo.boxw + lane];
                if (t0 + i >= S) v = q_zero();
                loc = q_mul(v, loc);
            }
            s_seg[seg][lane] = loc;
            __syncthreads();
            float4 Lc = q_ident();
            if (seg == 0) {
#pragma unroll
                for (int k = 0; k < NSEG; ++k) Lc = q_mul(s_seg[k][lane], Lc);
                if (chunk > 0 && item != ctl.stall_item)
                    publish1(arr.a_agg, arr.a_flags + idx, idx, lane, Lc, pack_flag(epoch, ST_AGG));
            }
            float4 carry = init_v;
            if (chunk > 0)
                carry = lookback_prod(arr.a_flags, arr.a_agg, arr.a_incl, chunk, g, NG, init_v, epoch, ctl, item,
                                      seg, lane, reinterpret_cast<float4(*)[LT]>(&s_lb[0][0][0]), s_st, &s_done);
            if (seg == 0 && item != ctl.stall_item)
                publish1(arr.a_incl, arr.a_flags + idx, idx, lane, q_mul(Lc, carry), pack_flag(epoch, ST_INCL));
        } else {
            // ---- C item: cotangents of this chunk ------------------------------
            // Forward local pass: lp[i] = product of the segment's steps before i,
            // W = sum_i conj(local_i) (x) d_cum[t0+i].
            float4 lp[N];
            float4 loc = q_ident(), W = q_zero();
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const int row = seg * N + i;
                float4 qv = Qt[row * geo.boxw + lane], dv = Dt[row * geo.boxw + lane];
                if (t0 + i >= S) {
                    qv = q_zero();
                    dv = q_zero();
                }
                lp[i] = loc;
                loc = q_mul(qv, loc);
                W = q_add(W, q_mul_cl(loc, dv));
            }
            s_seg[seg][lane] = loc;
            s_w[seg][lane] = W;
            __syncthreads();

            float4 Mt = q_ident(), Vt = q_zero();
            if (seg == 0) {
                // Suffix maps: segment k receives H = V_k + M_k (x) H_{chunk+1}.
                float4 M = q_ident(), V = q_zero();
#pragma unroll
                for (int k = NSEG - 1; k >= 0; --k) {
                    const float4 Lk = s_seg[k][lane], Wk = s_w[k][lane];
                    s_m[k][lane] = M;
                    s_w[k][lane] = V;
                    V = q_add(Wk, q_mul_cl(Lk, V));
                    M = q_mul_cl(Lk, M);
                }
                Mt = M;   // conj(L_c)
                Vt = V;   // W_c
                // Exclusive forward prefixes of the segment products (in place).
                float4 e = q_ident();
#pragma unroll
                for (int k = 0; k < NSEG; ++k) {
                    const float4 a = s_seg[k][lane];
                    s_seg[k][lane] = e;
                    e = q_mul(a, e);
                }
                if (chunk < C - 1 && item != ctl.stall_item)
                    publish2(arr.c_agg, arr.c_flags + idx, idx, lane, Mt, Vt, pack_flag(epoch, ST_AGG));
            }
            float4 Hnext = q_zero();
            if (chunk < C - 1)
                Hnext = lookback_affine(arr.c_flags, arr.c_agg, arr.c_incl, chunk, C, g, NG, epoch, ctl, item,
                                        seg, lane, s_lb, s_st, &s_done);
            if (seg == 0) {
                const float4 Hc = q_add(Vt, q_mul(Mt, Hnext));
                if (item != ctl.stall_item)
                    publish1(arr.c_incl, arr.c_flags + idx, idx, lane, Hc, pack_flag(epoch, ST_INCL));
                if (chunk == 0 && lane_ok) d_init[static_cast<long long>(b) * HJ + hj] = Hc;
                float4 F = init_v;
                if (chunk > 0) {
                    const long long aidx = idx - NG;   // A item of chunk - 1
                    bool failed = false;
                    wait_flag(arr.a_flags + aidx, epoch, ctl, item, ST_INCL, failed);
                    F = failed ? q_nan() : __ldcg(arr.a_incl + aidx * LT + lane);
                }
                s_carry[lane] = F;
                s_h[lane] = Hnext;
            }
            __syncthreads();

            // Reverse pass: G = d_cum + H_next, d_q = G (x) conj(cum[t-1]),
            // H = conj(q_t) (x) G handed to step t-1.
            const float4 X = q_mul(s_seg[seg][lane], s_carry[lane]);
            float4 Hn = q_add(s_w[seg][lane], q_mul(s_m[seg][lane], s_h[lane]));
            float4 *out = d_q + (static_cast<long long>(b) * S + t0) * HJ + hj;
#pragma unroll
            for (int i = N - 1; i >= 0; --i) {
                const int row = seg * N + i;
                float4 qv = Qt[row * geo.boxw + lane], dv = Dt[row * geo.boxw + lane];
                const bool t_ok = t0 + i < S;
                if (!t_ok) {
                    qv = q_zero();
                    dv = q_zero();
                }
                const float4 G = q_add(dv, Hn);
                const float4 cp = q_mul(lp[i], X);
                if (lane_ok && t_ok) __stcs(out + static_cast<long long>(i) * HJ, q_mul_cr(G, cp));
                Hn = q_mul_cl(qv, G);
            }
        }
        __syncthreads();
        head = (head + 1) % NST;
    }
    finish_launch(ctl, epoch);
}

}  // namespace qs

// ===========================================================================
// Host side: argument checks, workspace, tensor maps, launches, C ABI.
// ===========================================================================
namespace {

using qs::LT;
using qs::NSEG;
using qs::NTHREADS;

// Kernel variants (steps per thread N, pipeline stages NST).
constexpr int FWD_N = 8, FWD_NST = 2;
constexpr int BWD_N = 4, BWD_NST = 2;
constexpr int FWD_T = NSEG * FWD_N;
constexpr int BWD_T = NSEG * BWD_N;
constexpr size_t FWD_SMEM = size_t(FWD_NST) * FWD_T * LT * 16 + 1024;
constexpr size_t BWD_SMEM = size_t(BWD_NST) * 2 * BWD_T * LT * 16 + 1024;
// Target bytes of q per backward batch: small enough that the batch's q is
// still in L2 when its C items re-read it.
constexpr long long BWD_BATCH_Q_BYTES = 24ll << 20;
long long g_batch_q_bytes = BWD_BATCH_Q_BYTES;
constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;

std::mutex g_mu;
unsigned long long g_timeout_ns = DEFAULT_TIMEOUT_NS;
int g_stall_item = -1;

struct DevInfo {
    int sms = 0;
    int major = 0, minor = 0;
    int fwd_blocks = 0, bwd_blocks = 0;   // resident CTAs per SM
};
std::map<int, DevInfo> g_dev;

struct Workspace {
    unsigned char *base = nullptr;
    size_t bytes = 0;
};
std::map<std::pair<int, uintptr_t>, Workspace> g_ws;

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
            auto fk = qs::quat_scan_fwd_kernel<FWD_N, FWD_NST>;
            auto bk = qs::quat_scan_bwd_kernel<BWD_N, BWD_NST>;
            if (cudaFuncSetAttribute(fk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FWD_SMEM) != cudaSuccess ||
                cudaFuncSetAttribute(bk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BWD_SMEM) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.fwd_blocks, fk, NTHREADS, FWD_SMEM) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.bwd_blocks, bk, NTHREADS, BWD_SMEM) != cudaSuccess) {
                cudaGetLastError();
                d.sms = 0;
                return QS_ERR_CUDA;
            }
            d.fwd_blocks = std::max(d.fwd_blocks, 1);
            d.bwd_blocks = std::max(d.bwd_blocks, 1);
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
    qs::WsHeader h;
    std::memset(&h, 0, sizeof h);
    h.epoch = 1;
    if (cudaMemsetAsync(p, 0, bytes, stream) != cudaSuccess ||
        cudaMemcpyAsync(p, &h, sizeof h, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
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

// 3-D view [B][S][HJ*4 floats] of a [B,S,H,J,4] tensor; box = boxw lanes x boxh steps.
int make_map(CUtensorMap *m, const float *ptr, int64_t B, int64_t S, int64_t HJ, int boxw, int boxh) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return QS_ERR_CUDA;
    cuuint64_t dims[3] = {(cuuint64_t)(HJ * 4), (cuuint64_t)S, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)(HJ * 16), (cuuint64_t)(S * HJ * 16)};
    cuuint32_t box[3] = {(cuuint32_t)(boxw * 4), (cuuint32_t)boxh, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? QS_OK : QS_ERR_CUDA;
}

qs::Geometry geometry(int64_t B, int64_t S, int64_t HJ, int T) {
    qs::Geometry g;
    g.S = S;
    g.HJ = (int)HJ;
    g.NGb = (int)((HJ + LT - 1) / LT);
    g.NG = (int)(B * g.NGb);
    g.C = (int)((S + T - 1) / T);
    g.boxw = (int)std::min<int64_t>(LT, HJ);
    g.boxh = (int)std::min<int64_t>(T, S);
    return g;
}

qs::Schedule bwd_schedule(const qs::Geometry &g) {
    qs::Schedule s;
    s.CA = g.C - 1;
    const long long q_per_group = (long long)LT * g.S * 16;
    long long batch_bytes;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        batch_bytes = g_batch_q_bytes;
    }
    long long gb = batch_bytes / std::max<long long>(q_per_group, 1);
    gb = std::max<long long>(1, std::min<long long>(gb, g.NG));
    s.GB = (int)gb;
    s.NB = (g.NG + s.GB - 1) / s.GB;
    return s;
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

    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;

    const qs::Geometry geo = geometry(B, S, HJ, FWD_T);
    const long long nitems = (long long)geo.C * geo.NG;
    if (nitems >= (1ll << 31) - (1 << 20)) return QS_ERR_DIMS;
    size_t off = sizeof(qs::WsHeader);
    const size_t o_flags = off;
    off = align_up(off + nitems * 8, 256);
    const size_t o_agg = off;
    off = align_up(off + nitems * LT * 16, 256);
    const size_t o_incl = off;
    off = align_up(off + nitems * LT * 16, 256);
    unsigned char *ws = nullptr;
    rc = ensure_workspace(dev, stream, off, &ws);
    if (rc != QS_OK) return rc;

    CUtensorMap qmap;
    rc = make_map(&qmap, q, B, S, HJ, geo.boxw, geo.boxh);
    if (rc != QS_OK) return rc;

    qs::Control ctl;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ctl.timeout_ns = g_timeout_ns;
        ctl.stall_item = g_stall_item;
    }
    ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
    ctl.nitems = (int)nitems;
    const int grid = (int)std::min<long long>(nitems, (long long)di->sms * di->fwd_blocks);
    qs::quat_scan_fwd_kernel<FWD_N, FWD_NST><<<grid, NTHREADS, FWD_SMEM, stream>>>(
        qmap, reinterpret_cast<const float4 *>(init), reinterpret_cast<float4 *>(cum),
        reinterpret_cast<unsigned long long *>(ws + o_flags), reinterpret_cast<float4 *>(ws + o_agg),
        reinterpret_cast<float4 *>(ws + o_incl), geo, ctl);
    if (cudaGetLastError() != cudaSuccess) return QS_ERR_CUDA;
    return QS_OK;
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

    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;

    const qs::Geometry geo = geometry(B, S, HJ, BWD_T);
    const qs::Schedule sch = bwd_schedule(geo);
    const long long nA = (long long)sch.CA * geo.NG, nC = (long long)geo.C * geo.NG;
    const long long nitems = nA + nC;
    if (nitems >= (1ll << 31) - (1 << 20)) return QS_ERR_DIMS;
    size_t off = sizeof(qs::WsHeader);
    const size_t o_af = off;
    off = align_up(off + nA * 8, 256);
    const size_t o_aa = off;
    off = align_up(off + nA * LT * 16, 256);
    const size_t o_ai = off;
    off = align_up(off + nA * LT * 16, 256);
    const size_t o_cf = off;
    off = align_up(off + nC * 8, 256);
    const size_t o_ca = off;
    off = align_up(off + nC * LT * 32, 256);
    const size_t o_ci = off;
    off = align_up(off + nC * LT * 16, 256);
    unsigned char *ws = nullptr;
    rc = ensure_workspace(dev, stream, off, &ws);
    if (rc != QS_OK) return rc;

    CUtensorMap qmap, dmap;
    rc = make_map(&qmap, q, B, S, HJ, geo.boxw, geo.boxh);
    if (rc == QS_OK) rc = make_map(&dmap, d_cum, B, S, HJ, geo.boxw, geo.boxh);
    if (rc != QS_OK) return rc;

    qs::BwdArrays arr;
    arr.a_flags = reinterpret_cast<unsigned long long *>(ws + o_af);
    arr.a_agg = reinterpret_cast<float4 *>(ws + o_aa);
    arr.a_incl = reinterpret_cast<float4 *>(ws + o_ai);
    arr.c_flags = reinterpret_cast<unsigned long long *>(ws + o_cf);
    arr.c_agg = reinterpret_cast<float4 *>(ws + o_ca);
    arr.c_incl = reinterpret_cast<float4 *>(ws + o_ci);
    qs::Control ctl;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ctl.timeout_ns = g_timeout_ns;
        ctl.stall_item = g_stall_item;
    }
    ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
    ctl.nitems = (int)nitems;
    const int grid = (int)std::min<long long>(nitems, (long long)di->sms * di->bwd_blocks);
    qs::quat_scan_bwd_kernel<BWD_N, BWD_NST><<<grid, NTHREADS, BWD_SMEM, stream>>>(
        qmap, dmap, reinterpret_cast<const float4 *>(init), reinterpret_cast<float4 *>(d_q),
        reinterpret_cast<float4 *>(d_init), arr, geo, sch, ctl);
    if (cudaGetLastError() != cudaSuccess) return QS_ERR_CUDA;
    return QS_OK;
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
    const size_t o = offsetof(qs::WsHeader, err_code);
    if (cudaMemset(base + o, 0, 2 * sizeof(unsigned int)) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    return QS_ERR_TIMEOUT;
}

extern "C" const char *quat_cumprod_strerror(int status) {
    switch (status) {
        case QS_OK: return "success";
        case QS_ERR_NULL: return "a required pointer is NULL";
        case QS_ERR_DIMS: return "a size is negative or beyond the supported limits";
        case QS_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
        case QS_ERR_ALIAS: return "an output overlaps an input";
        case QS_ERR_CUDA: return "a CUDA runtime call failed";
        case QS_ERR_TIMEOUT: return "a cross-tile wait on the device ran out (outputs are invalid)";
        case QS_ERR_NOMEM: return "workspace allocation failed or would be needed during stream capture";
        case QS_ERR_DEVICE: return "the current device is not compute capability 10.3 (sm_103)";
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
    g_stall_item = (tile < 0 || tile > INT32_MAX) ? -1 : (int)tile;
    return QS_OK;
}

extern "C" int quat_cumprod_debug_set_batch_bytes(int64_t bytes) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_batch_q_bytes = bytes > 0 ? (long long)bytes : BWD_BATCH_Q_BYTES;
    return QS_OK;
}

// Host-side check of the backward work-item schedule for these sizes: every
// (phase, chunk, group) item appears exactly once, A items of a group come in
// increasing chunk order, C items in decreasing chunk order, and the A item of
// chunk c precedes the C item of chunk c+1 (the only cross-phase wait).
extern "C" int quat_cumprod_debug_check_schedule(int64_t B, int64_t S, int64_t H, int64_t J) {
    const int dc = check_dims(B, S, H, J);
    if (dc == 1) return QS_OK;
    if (dc != QS_OK) return dc;
    const qs::Geometry geo = geometry(B, S, H * J, BWD_T);
    const qs::Schedule sch = bwd_schedule(geo);
    const long long nA = (long long)sch.CA * geo.NG, nC = (long long)geo.C * geo.NG;
    if (nA + nC > (1ll << 26)) return QS_ERR_DIMS;   // keep the check cheap
    std::vector<int> posA(nA > 0 ? nA : 1, -1), posC(nC, -1);
    for (long long id = 0; id < nA + nC; ++id) {
        const qs::Work w = qs::decode_bwd((int)id, geo.NG, geo.C, sch);
        if (w.g < 0 || w.g >= geo.NG || w.chunk < 0) return -100;
        if (w.phase == 0) {
            if (w.chunk >= sch.CA) return -101;
            int &p = posA[(long long)w.chunk * geo.NG + w.g];
            if (p != -1) return -102;
            p = (int)id;
        } else {
            if (w.chunk >= geo.C) return -103;
            int &p = posC[(long long)w.chunk * geo.NG + w.g];
            if (p != -1) return -104;
            p = (int)id;
        }
    }
    for (int g = 0; g < geo.NG; ++g) {
        for (int c = 0; c < geo.C; ++c) {
            const int pc = posC[(long long)c * geo.NG + g];
            if (pc < 0) return -105;
            if (c + 1 < geo.C && posC[(long long)(c + 1) * geo.NG + g] > pc) return -106;
            if (c < sch.CA) {
                const int pa = posA[(long long)c * geo.NG + g];
                if (pa < 0) return -107;
                if (c > 0 && posA[(long long)(c - 1) * geo.NG + g] > pa) return -108;
                if (pa > posC[(long long)(c + 1) * geo.NG + g]) return -109;
            }
        }
    }
    return QS_OK;
}
