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
//  * Tile = LT lanes x T consecutive steps of one lane group (LT lanes of one
//    batch entry, contiguous in memory), staged into shared memory by 3-D TMA
//    loads of boxes of up to 64 lanes.  Compute thread (seg, lane) owns N
//    consecutive steps of one lane; NSEG = 256 / LT segments per tile.
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
//  * One persistent kernel per direction runs three kinds of work items from
//    one global queue:
//      P1 (chunk, group): read the tile, publish L_c (and W_c);
//      SC (group, 32-lane block): once all P1 items of the group are published,
//                         scan its chunk aggregates (8 threads per lane) into
//                         the carries F_c (and H_{c+1}, and d_init);
//      P3 (chunk, group): read the tile again, apply the carries, write cum (or
//                         d_q) into shared memory, store it with TMA.
//    Lane groups are processed in batches whose inputs fit the L2 cache; the
//    queue runs P1(0) SC(0) | P1(1) SC(1) P3(0) | P1(2) SC(2) P3(1) | ... so
//    the P3 pass of a batch re-reads its tiles from L2.
//
//  * Warp roles inside a CTA (10 warps): 8 compute warps run the items; a
//    producer warp claims items, issues TMA loads several stages ahead and
//    fetches the carries of P3 items; a publisher warp writes P1 aggregates
//    out (fence, flag), issues the TMA stores of P3 outputs and frees stages.
//    They hand stages over through mbarriers (full / done / empty), so no
//    global-memory latency sits on the compute warps' path.
//
//  * Every cross-CTA wait is on an item claimed earlier from the queue (no
//    deadlock) and is bounded in time: it reports QS_ERR_TIMEOUT instead of
//    hanging.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "quat_cumprod.h"
#include "quat_device.cuh"

namespace qs {

constexpr int NCOMPUTE = 256;            // compute threads per CTA (8 warps)
constexpr int PRODUCER_WARP = 8;
constexpr int PUBLISHER_WARP = 9;
constexpr int NTHREADS = NCOMPUTE + 64;  // + producer warp + publisher warp
constexpr int CLAIM = 4;                 // items claimed per atomic

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
};

struct Control {
    WsHeader *hdr;
    int nitems;
    int stall_item;
    unsigned long long timeout_ns;
    int ctr_cap;   // entries of each P1 counter array
};

struct Arrays {
    unsigned int *p1_count;         // [2][ctr_cap] P1 items published per lane group;
                                    // array (epoch & 1) counts this launch, the other
                                    // one is cleared for the next launch
    unsigned long long *sc_flags;   // [NG*NSB]     SC item published
    float4 *aggL;                   // [C*NG*LT] chunk product L_c
    float4 *aggW;                   // [C*NG*LT] chunk weighted sum W_c (backward)
    float4 *carF;                   // [C*NG*LT] forward carry cum[t0-1]
    float4 *carH;                   // [C*NG*LT] H entering the chunk from the right (backward)
};

// Batches of lane groups: batch k holds groups [k*GB, k*GB + gk).
struct Schedule {
    int GB;    // lane groups per batch
    int NB;    // batches
    int NSB;   // 32-lane blocks per group (SC items per group)
};

enum : int { KIND_P1 = 0, KIND_SC = 1, KIND_P3 = 2 };

struct Work {
    int kind;
    int chunk;   // P1/P3
    int g;       // lane group
    int sb;      // 32-lane block (SC)
};

// Queue order: block 0 = P1(0) SC(0); block k (1..NB-1) = P1(k) SC(k) P3(k-1);
// block NB = P3(NB-1).  Inside P1/P3 of a batch: chunk-major (all groups of
// the batch at chunk c, then chunk c+1).  Item counts stay below 2^31, so the
// arithmetic is 32-bit.
__host__ __device__ inline Work decode_item(int id, int NG, int C, const Schedule &s) {
    const unsigned uC = static_cast<unsigned>(C), GB = static_cast<unsigned>(s.GB);
    const unsigned NSB = static_cast<unsigned>(s.NSB);
    const unsigned last_g = static_cast<unsigned>(NG - (s.NB - 1) * s.GB);
    const unsigned g0 = (s.NB == 1) ? last_g : GB;
    const unsigned b0 = uC * g0 + g0 * NSB;
    unsigned r = static_cast<unsigned>(id), local;
    int k, kind;
    if (r < b0) {
        k = 0;
        if (r < uC * g0) {
            kind = KIND_P1;
            local = r;
        } else {
            kind = KIND_SC;
            local = r - uC * g0;
        }
    } else {
        r -= b0;
        const unsigned full = 2u * uC * GB + GB * NSB;   // block with full P1, SC, P3
        const unsigned nfull = s.NB > 2 ? static_cast<unsigned>(s.NB - 2) : 0u;   // blocks 1..NB-2
        if (r < nfull * full) {
            const unsigned blk = 1u + r / full;
            r -= (blk - 1u) * full;
            if (r < uC * GB) {
                kind = KIND_P1;
                k = static_cast<int>(blk);
                local = r;
            } else if (r < uC * GB + GB * NSB) {
                kind = KIND_SC;
                k = static_cast<int>(blk);
                local = r - uC * GB;
            } else {
                kind = KIND_P3;
                k = static_cast<int>(blk) - 1;
                local = r - uC * GB - GB * NSB;
            }
        } else {
            r -= nfull * full;
            if (s.NB >= 2) {
                // block NB-1: P1(NB-1) [C*last_g], SC(NB-1) [last_g*NSB], P3(NB-2) [C*GB]
                const unsigned a1 = uC * last_g, a2 = a1 + last_g * NSB, a3 = a2 + uC * GB;
                if (r < a1) {
                    kind = KIND_P1;
                    k = s.NB - 1;
                    local = r;
                } else if (r < a2) {
                    kind = KIND_SC;
                    k = s.NB - 1;
                    local = r - a1;
                } else if (r < a3) {
                    kind = KIND_P3;
                    k = s.NB - 2;
                    local = r - a2;
                } else {
                    kind = KIND_P3;
                    k = s.NB - 1;
                    local = r - a3;
                }
            } else {
                kind = KIND_P3;
                k = 0;
                local = r;
            }
        }
    }
    const unsigned gk = (k == s.NB - 1) ? last_g : GB;
    Work w;
    w.kind = kind;
    if (kind == KIND_SC) {
        w.chunk = 0;
        w.g = k * s.GB + static_cast<int>(local / NSB);
        w.sb = static_cast<int>(local - (local / NSB) * NSB);
    } else {
        const unsigned c = local / gk;
        w.chunk = static_cast<int>(c);
        w.g = k * s.GB + static_cast<int>(local - c * gk);
        w.sb = 0;
    }
    return w;
}

__device__ __forceinline__ unsigned long long pack_flag(uint32_t epoch) {
    return static_cast<unsigned long long>(epoch);
}

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
    return reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ void record_error(WsHeader *h, uint32_t epoch, int item) {
    if (atomicCAS(&h->err_code, 0u, 1u) == 0u) h->err_item = static_cast<unsigned long long>(item);
    atomicAdd(&h->err_count, 1u);
    atomicExch(&h->err_epoch, epoch);
}

// True once this launch has recorded a timeout: every wait then gives up at
// once so that the launch drains quickly (its outputs are invalid anyway).
__device__ __forceinline__ bool launch_failed(const Control &ctl, uint32_t epoch) {
    return ld_volatile_u32(&ctl.hdr->err_epoch) == epoch;
}

// Waits until the flags base[c*stride] for c = begin, begin+step, ... < end all
// carry this launch's epoch.  The flags are polled with relaxed loads issued
// eight at a time and acquired by one fence once all have been seen.  Bounded:
// gives up after ctl.timeout_ns (records the error) or as soon as another CTA
// of this launch has given up.  Returns false if it gave up.
__device__ __noinline__ bool wait_flags(const unsigned long long *base, long long stride, int begin, int end,
                                        int step, uint32_t epoch, const Control &ctl, int item) {
    const unsigned long long want = pack_flag(epoch);
    unsigned long long t0 = 0;
    unsigned ns = 32;
    int c = begin;
    for (int round = 0;; ++round) {
        while (c < end) {
            unsigned long long f[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int cc = c + u * step;
                f[u] = cc < end ? ld_relaxed_u64(base + cc * stride) : want;
            }
            int ready = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (f[u] != want) break;
                ++ready;
            }
            c += ready * step;
            if (ready < 8) break;
        }
        if (c >= end) {
            fence_acquire_gpu();
            return true;
        }
        if (round == 0) t0 = global_timer_ns();
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
        if (launch_failed(ctl, epoch)) return false;
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            record_error(ctl.hdr, epoch, item);
            return false;
        }
    }
}

// Waits until the counter reaches `target` (relaxed polling, then one acquire
// fence); bounded like wait_flags.
__device__ __noinline__ bool wait_count(const unsigned int *ctr, unsigned target, uint32_t epoch,
                                        const Control &ctl, int item) {
    unsigned long long t0 = 0;
    unsigned ns = 32;
    for (int round = 0;; ++round) {
        unsigned v;
        asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) {
            fence_acquire_gpu();
            return true;
        }
        if (round == 0) t0 = global_timer_ns();
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
        if (launch_failed(ctl, epoch)) return false;
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            record_error(ctl.hdr, epoch, item);
            return false;
        }
    }
}

// Waits for a phase of an intra-CTA mbarrier.  These phases depend only on
// this CTA's own warps and TMA copies, so they complete unless something is
// broken; the wait is still bounded (records the error, returns false).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, unsigned long long limit_ns,
                                         const Control &ctl, uint32_t epoch, int item) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            record_error(ctl.hdr, epoch, item);
            return false;
        }
    }
    return true;
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

// Shared-memory footprint of one kernel configuration (dynamic part).
__host__ __device__ constexpr size_t smem_bytes(bool bwd, int lt, int n, int nst) {
    return 1024                                                        // alignment slack
           + size_t(nst) * (bwd ? 2 : 1) * (NCOMPUTE / lt) * n * lt * 16  // stages
           + size_t(nst) * (bwd ? 2 : 1) * lt * 16                      // per-stage result / carry slot
           + size_t(2) * NCOMPUTE * 16 * (bwd ? 2 : 1);                  // segment results (2 parities)
}

// ---------------------------------------------------------------------------
// The scan kernel.  BWD = false: forward (q -> cum).  BWD = true: backward
// ((q, d_cum) -> (d_q, d_init)).
// ---------------------------------------------------------------------------
template <bool BWD, int LT, int N, int NST>
__global__ void __launch_bounds__(NTHREADS, 1)
    quat_scan_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap dmap,
                     const __grid_constant__ CUtensorMap omap, const float4 *__restrict__ init,
                     float4 *__restrict__ d_init, const Arrays arr, const Geometry geo, const Schedule sch,
                     const Control ctl) {
    static_assert(NST >= 3, "at least three stages");
    static_assert(LT == 32 || LT == 64 || LT == 128, "lane group width");
    constexpr int NSEG = NCOMPUTE / LT;
    constexpr int T = NSEG * N;
    static_assert(T <= 256, "TMA box height");
    static_assert(smem_bytes(BWD, LT, N, NST) <= 226 * 1024, "shared memory per CTA");
    // One TMA box per operand: [T rows][LT lanes], row-major.  128-lane groups
    // use a 4-D view (64-lane blocks), narrower groups a 3-D view.
    constexpr bool MAP4 = LT == 128;
    constexpr uint32_t HALF = T * LT * 16;                  // one operand of a stage
    constexpr uint32_t STAGE = BWD ? 2 * HALF : HALF;
    constexpr int NRES = BWD ? 2 : 1;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = align1024(smem_raw);
    // [stages][P1 results][P3 carries][segment results]
    // Per-stage slot: the P1 results of a stage's item (compute -> publisher),
    // or the carries of its P3 item (producer -> compute).
    float4 *s_rc = reinterpret_cast<float4 *>(smem + size_t(NST) * STAGE);        // [NST][NRES][LT]
    float4 *s_seg = s_rc + NST * NRES * LT;                                       // [2][NRES][NSEG][LT]
    __shared__ __align__(8) uint64_t full_bar[NST], done_bar[NST], empty_bar[NST];
    __shared__ int s_items[NST];
    __shared__ int4 s_work[NST];   // decoded item: kind, chunk, group, 32-lane block
    __shared__ int s_end_seq;
    __shared__ int s_abort;   // set when an intra-CTA wait ran out: every role stops

    const int tid = threadIdx.x, warp = tid >> 5, wl = tid & 31;
    const uint32_t epoch = ld_volatile_u32(&ctl.hdr->epoch);
    const int HJ = geo.HJ, NG = geo.NG, C = geo.C;
    const unsigned long long flag_val = pack_flag(epoch);

    {   // clear the other counter array for the next launch on this workspace
        unsigned int *next = arr.p1_count + ((epoch + 1u) & 1u) * ctl.ctr_cap;
        for (int i = blockIdx.x * NTHREADS + tid; i < ctl.ctr_cap; i += gridDim.x * NTHREADS) next[i] = 0u;
    }
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full_bar[s], 2);                 // issue + fetch
            mbar_init(&done_bar[s], NCOMPUTE / 32);     // one per compute warp
            mbar_init(&empty_bar[s], 1);                // publisher
        }
        s_end_seq = -1;
        s_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();


    if (warp == PRODUCER_WARP) {
        // ================= producer: claims, TMA loads, carries =================
        if (wl == 0) {
            prefetch_tensormap(&qmap);
            if (BWD) prefetch_tensormap(&dmap);
        }
        int seq_issue = 0, seq_fetch = 0, claim_next = 0, claim_left = 0;
        bool ended = false;
        unsigned long long idle_since = 0, stuck_since = 0;
        int spins = 0;
        for (;;) {
            if (*reinterpret_cast<volatile int *>(&s_abort)) break;
            bool prog = false;
            // -- issue items into free stages --
            while (!ended) {
                const int s = seq_issue % NST;
                const bool free_stage =
                    seq_issue < NST || mbar_test_wait(&empty_bar[s], ((seq_issue / NST) - 1) & 1);
                if (!free_stage) break;
                {
                    if (claim_left == 0) {
                        int c0 = 0;
                        if (wl == 0) c0 = static_cast<int>(atomicAdd(&ctl.hdr->counter, (unsigned)CLAIM));
                        claim_next = __shfl_sync(0xffffffffu, c0, 0);
                        claim_left = CLAIM;
                    }
                    const int it = claim_next++;
                    --claim_left;
                    if (it >= ctl.nitems) {
                        ended = true;
                        if (wl == 0) {
                            s_items[s] = -1;
                            s_end_seq = seq_issue;
                            mbar_arrive(&full_bar[s]);
                            mbar_arrive(&full_bar[s]);
                        }
                    } else {
                        const Work w = decode_item(it, NG, C, sch);
                        if (wl == 0) {
                            s_items[s] = it;
                            s_work[s] = make_int4(w.kind, w.chunk, w.g, w.sb);
                            if (w.kind == KIND_SC) {
                                mbar_arrive(&full_bar[s]);
                            } else {
                                const int b = w.g / geo.NGb, gx = w.g - b * geo.NGb;
                                unsigned char *dst = smem + size_t(s) * STAGE;
                                mbar_arrive_expect_tx(&full_bar[s], STAGE);
                                if (MAP4) {
                                    tma_load_4d(dst, &qmap, 0, gx * 2, w.chunk * T, b, &full_bar[s]);
                                    if (BWD) tma_load_4d(dst + HALF, &dmap, 0, gx * 2, w.chunk * T, b, &full_bar[s]);
                                } else {
                                    tma_load_3d(dst, &qmap, gx * LT * 4, w.chunk * T, b, &full_bar[s]);
                                    if (BWD) tma_load_3d(dst + HALF, &dmap, gx * LT * 4, w.chunk * T, b, &full_bar[s]);
                                }
                            }
                        }
                        ++seq_issue;
                    }
                    __syncwarp();
                    prog = true;
                }
            }
            // -- complete the next issued item: carries of P3 items --
            if (seq_fetch < seq_issue) {
                const int s = seq_fetch % NST;
                const int it = s_items[s];
                const int4 wk = s_work[s];
                const Work w{wk.x, wk.y, wk.z, wk.w};
                bool ready = true;
                if (w.kind == KIND_P3) {
                    // all 32-lane blocks of the group must have been scanned
                    const unsigned long long f =
                        wl < sch.NSB ? ld_relaxed_u64(arr.sc_flags + static_cast<long long>(w.g) * sch.NSB + wl)
                                     : flag_val;
                    ready = __all_sync(0xffffffffu, f == flag_val);
                    bool give_up = false;
                    if (!ready && spins > 64) {
                        if (idle_since == 0) idle_since = global_timer_ns();
                        if (launch_failed(ctl, epoch)) give_up = true;
                        else if (global_timer_ns() - idle_since > ctl.timeout_ns) {
                            if (wl == 0) record_error(ctl.hdr, epoch, it);
                            give_up = true;
                        }
                    }
                    if (ready || give_up) {
                        fence_acquire_gpu();
                        const long long base = (static_cast<long long>(w.chunk) * NG + w.g) * LT;
                        for (int l = wl; l < LT; l += 32) {
                            s_rc[(s * NRES + 0) * LT + l] = give_up ? q_nan() : __ldcg(arr.carF + base + l);
                            if (BWD) s_rc[(s * NRES + 1) * LT + l] = give_up ? q_nan() : __ldcg(arr.carH + base + l);
                        }
                        ready = true;
                        idle_since = 0;
                    }
                }
                if (ready) {
                    __syncwarp();
                    if (wl == 0) mbar_arrive(&full_bar[s]);
                    ++seq_fetch;
                    prog = true;
                }
            }
            if (ended && seq_fetch == seq_issue) break;
            if (prog) {
                spins = 0;
                stuck_since = 0;
            } else {
                ++spins;
                __nanosleep(32);
                if ((spins & 255) == 0) {
                    const unsigned long long now = global_timer_ns();
                    if (stuck_since == 0) {
                        stuck_since = now;
                    } else if (now - stuck_since > 4 * ctl.timeout_ns) {
                        if (wl == 0) {
                            record_error(ctl.hdr, epoch, -1);
                            s_abort = 1;
                        }
                        __syncwarp();
                        break;
                    }
                }
            }
        }
        // Never leave with TMA loads in flight: complete the second arrival of
        // issued items that were not fetched, then wait (bounded) for every
        // stage's last issued phase.
        if (*reinterpret_cast<volatile int *>(&s_abort) && wl == 0) {
            for (int q = seq_fetch; q < seq_issue; ++q) mbar_arrive(&full_bar[q % NST]);
            for (int q = seq_issue - NST; q < seq_issue; ++q)
                if (q >= 0) wait_bar(&full_bar[q % NST], (q / NST) & 1, 10000000ull, ctl, epoch, -1);
        }
    } else if (warp == PUBLISHER_WARP) {
        // ================= publisher: P1 aggregates, P3 stores, free stages =====
        if (wl == 0) prefetch_tensormap(&omap);
        unsigned int *cnt = arr.p1_count + (epoch & 1u) * ctl.ctr_cap;
        int pend[NST + 1];   // lane groups of P1 items written but not yet counted
        int npend = 0;
        // One fence makes every aggregate written so far visible, then each
        // pending P1 item is counted for its lane group.
        auto flush_pending = [&]() {
            if (npend == 0) return;
            __threadfence();
            __syncwarp();
            if (wl == 0)
                for (int k = 0; k < npend; ++k) atomicAdd(cnt + pend[k], 1u);
            npend = 0;
        };
        for (int seq = 0;; ++seq) {
            const int s = seq % NST;
            const uint32_t par = (seq / NST) & 1;
            bool have = false;
            unsigned long long t0 = 0;
            for (int spin = 0;; ++spin) {
                if (mbar_test_wait(&done_bar[s], par)) {
                    have = true;
                    break;
                }
                flush_pending();   // nothing else to do: publish what is pending
                if (*reinterpret_cast<volatile int *>(&s_end_seq) == seq) break;
                if (*reinterpret_cast<volatile int *>(&s_abort)) break;
                __nanosleep(32);
                if (spin == 64) t0 = global_timer_ns();
                if (spin > 64 && (spin & 63) == 0 && global_timer_ns() - t0 > 4 * ctl.timeout_ns) {
                    if (wl == 0) {
                        record_error(ctl.hdr, epoch, -1);
                        s_abort = 1;
                    }
                    break;
                }
            }
            if (!have) break;
            const int it = s_items[s];
            const int4 wk = s_work[s];
            const Work w{wk.x, wk.y, wk.z, wk.w};
            if (w.kind == KIND_P1) {
                const long long base = (static_cast<long long>(w.chunk) * NG + w.g) * LT;
                for (int l = wl; l < LT; l += 32) {
                    __stcg(arr.aggL + base + l, s_rc[(s * NRES + 0) * LT + l]);
                    if (BWD) __stcg(arr.aggW + base + l, s_rc[(s * NRES + 1) * LT + l]);
                }
                // Counted (and fenced) later, in a batch: see flush_pending.
                if (it != ctl.stall_item) pend[npend++] = w.g;
            } else if (w.kind == KIND_P3 && wl == 0) {
                const int b = w.g / geo.NGb, gx = w.g - b * geo.NGb;
                const unsigned char *src = smem + size_t(s) * STAGE + (BWD ? HALF : 0);
                if (MAP4)
                    tma_store_4d(&omap, src, 0, gx * 2, w.chunk * T, b);
                else
                    tma_store_3d(&omap, src, gx * LT * 4, w.chunk * T, b);
            }
            if (npend >= NST) flush_pending();
            if (wl == 0) {
                if (w.kind == KIND_P3) {
                    bulk_commit_group();
                    bulk_wait_group_read<0>();  // the store has read the stage
                }
                mbar_arrive(&empty_bar[s]);
            }
            __syncwarp();
        }
        flush_pending();
        if (wl == 0) bulk_wait_group_all();
    } else {
        // ================= compute warps =========================================
        const int ctid = tid;                  // 0..255
        const int lane = ctid % LT, seg = ctid / LT;
        for (int seq = 0;; ++seq) {
            const int s = seq % NST;
            const bool ok = wait_bar(&full_bar[s], (seq / NST) & 1, 4 * ctl.timeout_ns, ctl, epoch, -1);
            // All compute warps leave together if any wait ran out.
            if (named_bar_or(2, NCOMPUTE, !ok || *reinterpret_cast<volatile int *>(&s_abort))) {
                if (ctid == 0) s_abort = 1;
                break;
            }
            const int item = s_items[s];
            if (item < 0) break;
            const int4 wk = s_work[s];
            const Work w{wk.x, wk.y, wk.z, wk.w};
            const int par = seq & 1;
            float4 *sa = s_seg + (par * NRES + 0) * NCOMPUTE;      // [NSEG][LT]
            float4 *sw = s_seg + (par * NRES + (BWD ? 1 : 0)) * NCOMPUTE;
            float4 *Qt = reinterpret_cast<float4 *>(smem + size_t(s) * STAGE);
            float4 *Dt = reinterpret_cast<float4 *>(smem + size_t(s) * STAGE + HALF);
            const int cell0 = seg * N * LT + lane;   // this thread's first step

            if (w.kind == KIND_P1) {
                // ---- chunk aggregates --------------------------------------------
                float4 loc = q_ident(), W = q_zero();
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    loc = q_mul(Qt[cell0 + i * LT], loc);
                    if (BWD) W = q_add(W, q_mul_cl(loc, Dt[cell0 + i * LT]));
                }
                sa[seg * LT + lane] = loc;
                if (BWD) sw[seg * LT + lane] = W;
                named_bar_sync(1, NCOMPUTE);
                if (seg == 0) {
                    float4 L = q_ident();
#pragma unroll
                    for (int k = 0; k < NSEG; ++k) L = q_mul(sa[k * LT + lane], L);
                    s_rc[(s * NRES + 0) * LT + lane] = L;
                    if (BWD) {
                        float4 V = q_zero();
#pragma unroll
                        for (int k = NSEG - 1; k >= 0; --k) V = q_add(sw[k * LT + lane], q_mul_cl(sa[k * LT + lane], V));
                        s_rc[(s * NRES + 1) * LT + lane] = V;
                    }
                }
            } else if (w.kind == KIND_SC) {
                // ---- scan of one 32-lane block's chunk aggregates ----------------
                wait_count(arr.p1_count + (epoch & 1u) * ctl.ctr_cap + w.g, static_cast<unsigned>(C), epoch, ctl,
                           item);
                named_bar_sync(1, NCOMPUTE);
                constexpr int U = BWD ? 8 : 16;   // aggregates loaded per batch (independent loads)
                constexpr int RT = NCOMPUTE / 32;   // threads per lane (chunk ranges)
                const int sl = ctid & 31, rg = ctid >> 5;   // lane in the block, range
                const int l = w.sb * 32 + sl;               // lane in the group
                const int b = w.g / geo.NGb, hj = (w.g - b * geo.NGb) * LT + l;
                const bool lane_ok = hj < HJ;
                const int R = (C + RT - 1) / RT;
                const int c_lo = min(C, rg * R), c_hi = min(C, c_lo + R);
                auto at = [&](int c) { return (static_cast<long long>(c) * NG + w.g) * LT + l; };
                float4 *xa = sa;                       // [RT][32] range products
                float4 *xm = s_seg + (par ^ 1) * NRES * NCOMPUTE;   // [RT][32] (other parity is free here)
                float4 *xv = sw;
                float4 P = q_ident(), M = q_ident(), V = q_zero();
                for (int c0 = c_lo; c0 < c_hi; c0 += U) {
                    float4 Lb[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) Lb[u] = (c0 + u < c_hi) ? __ldcg(arr.aggL + at(c0 + u)) : q_ident();
#pragma unroll
                    for (int u = 0; u < U; ++u) P = q_mul(Lb[u], P);
                }
                if (BWD) {
                    for (int c1 = c_hi; c1 > c_lo; c1 -= U) {
                        float4 Lb[U], Wb[U];
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int c = c1 - 1 - u;
                            const bool in = c >= c_lo;
                            Lb[u] = in ? __ldcg(arr.aggL + at(c)) : q_ident();
                            Wb[u] = in ? __ldcg(arr.aggW + at(c)) : q_zero();
                        }
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            V = q_add(Wb[u], q_mul_cl(Lb[u], V));
                            M = q_mul_cl(Lb[u], M);
                        }
                    }
                }
                xa[rg * 32 + sl] = P;
                if (BWD) {
                    xm[rg * 32 + sl] = M;
                    xv[rg * 32 + sl] = V;
                }
                named_bar_sync(1, NCOMPUTE);
                float4 carry = lane_ok ? init[static_cast<long long>(b) * HJ + hj] : q_ident();
                for (int k = 0; k < rg; ++k) carry = q_mul(xa[k * 32 + sl], carry);
                float4 h = q_zero();
                if (BWD) {
                    for (int k = RT - 1; k > rg; --k) h = q_add(xv[k * 32 + sl], q_mul(xm[k * 32 + sl], h));
                    if (rg == 0 && lane_ok) d_init[static_cast<long long>(b) * HJ + hj] = q_add(V, q_mul(M, h));
                }
                for (int c0 = c_lo; c0 < c_hi; c0 += U) {
                    float4 Lb[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) Lb[u] = (c0 + u < c_hi) ? __ldcg(arr.aggL + at(c0 + u)) : q_ident();
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        if (c0 + u < c_hi) __stcg(arr.carF + at(c0 + u), carry);
                        carry = q_mul(Lb[u], carry);
                    }
                }
                if (BWD) {
                    for (int c1 = c_hi; c1 > c_lo; c1 -= U) {
                        float4 Lb[U], Wb[U];
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int c = c1 - 1 - u;
                            const bool in = c >= c_lo;
                            Lb[u] = in ? __ldcg(arr.aggL + at(c)) : q_ident();
                            Wb[u] = in ? __ldcg(arr.aggW + at(c)) : q_zero();
                        }
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int c = c1 - 1 - u;
                            if (c >= c_lo) __stcg(arr.carH + at(c), h);
                            h = q_add(Wb[u], q_mul_cl(Lb[u], h));
                        }
                    }
                }
                __threadfence();
                named_bar_sync(1, NCOMPUTE);
                if (ctid == 0 && item != ctl.stall_item)
                    st_release_u64(arr.sc_flags + static_cast<long long>(w.g) * sch.NSB + w.sb, flag_val);
            } else {
                // ---- apply the carries, write the outputs in place ---------------
                const float4 F = s_rc[(s * NRES + 0) * LT + lane];
                if (!BWD) {
                    float4 x[N];
                    float4 loc = q_ident();
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        loc = q_mul(Qt[cell0 + i * LT], loc);
                        x[i] = loc;
                    }
                    sa[seg * LT + lane] = loc;
                    named_bar_sync(1, NCOMPUTE);
                    float4 X = F;   // cum just before this segment
                    for (int k = 0; k < seg; ++k) X = q_mul(sa[k * LT + lane], X);
#pragma unroll
                    for (int i = 0; i < N; ++i) Qt[cell0 + i * LT] = q_mul(x[i], X);
                } else {
                    float4 lp[N];
                    float4 loc = q_ident(), W = q_zero();
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        lp[i] = loc;
                        loc = q_mul(Qt[cell0 + i * LT], loc);
                        W = q_add(W, q_mul_cl(loc, Dt[cell0 + i * LT]));
                    }
                    sa[seg * LT + lane] = loc;
                    sw[seg * LT + lane] = W;
                    named_bar_sync(1, NCOMPUTE);
                    float4 X = F;
                    for (int k = 0; k < seg; ++k) X = q_mul(sa[k * LT + lane], X);
                    float4 Hn = s_rc[(s * NRES + 1) * LT + lane];
                    for (int k = NSEG - 1; k > seg; --k) Hn = q_add(sw[k * LT + lane], q_mul_cl(sa[k * LT + lane], Hn));
                    // Reverse pass: G = d_cum + H, d_q = G (x) conj(cum[t-1]),
                    // H = conj(q_t) (x) G handed to step t-1.
#pragma unroll
                    for (int i = N - 1; i >= 0; --i) {
                        const float4 qv = Qt[cell0 + i * LT];
                        const float4 G = q_add(Dt[cell0 + i * LT], Hn);
                        Dt[cell0 + i * LT] = q_mul_cr(G, q_mul(lp[i], X));
                        Hn = q_mul_cl(qv, G);
                    }
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (wl == 0) mbar_arrive(&done_bar[s]);
        }
    }
    finish_launch(ctl, epoch);
}

}  // namespace qs

// ===========================================================================
// Host side: argument checks, workspace, tensor maps, launches, C ABI.
// ===========================================================================
namespace {

using qs::NTHREADS;

constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;
// Target input bytes per batch of lane groups (q for the forward, q + d_cum for
// the backward): about two batches plus the streamed outputs must stay in L2.
constexpr long long DEFAULT_BATCH_BYTES = 24ll << 20;

using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, const float4 *, float4 *, qs::Arrays,
                          qs::Geometry, qs::Schedule, qs::Control);

// One compiled configuration: lane-group width LT, steps per thread N, stages.
struct Variant {
    KernelFn fn;
    bool bwd;
    int lt, n, nstage;
    int T() const { return (qs::NCOMPUTE / lt) * n; }
    size_t smem() const { return qs::smem_bytes(bwd, lt, n, nstage); }
};

#define QS_VARIANT(B, LT, N, NS) \
    Variant { reinterpret_cast<KernelFn>(qs::quat_scan_kernel<B, LT, N, NS>), B, LT, N, NS }
// 128-lane configurations need H*J to be a multiple of 64 (4-D TMA view).
const Variant kFwdVariants[] = {
    QS_VARIANT(false, 128, 8, 6),   // 16-step chunks, 6 x 32 KiB stages
    QS_VARIANT(false, 64, 8, 6),    // 32-step chunks, 6 x 32 KiB stages
    QS_VARIANT(false, 32, 8, 6),    // 64-step chunks, 6 x 32 KiB stages
    QS_VARIANT(false, 128, 16, 3),  // 32-step chunks, 3 x 64 KiB stages
};
const Variant kBwdVariants[] = {
    QS_VARIANT(true, 64, 4, 6),     // 16-step chunks, 6 x 32 KiB stages
    QS_VARIANT(true, 32, 4, 6),     // 32-step chunks, 6 x 32 KiB stages
    QS_VARIANT(true, 128, 4, 5),    // 8-step chunks, 5 x 32 KiB stages
    QS_VARIANT(true, 64, 8, 3),     // 32-step chunks, 3 x 64 KiB stages
};
#undef QS_VARIANT
constexpr int kNumFwd = sizeof(kFwdVariants) / sizeof(kFwdVariants[0]);
constexpr int kNumBwd = sizeof(kBwdVariants) / sizeof(kBwdVariants[0]);

std::mutex g_mu;
unsigned long long g_timeout_ns = DEFAULT_TIMEOUT_NS;
int g_stall_item = -1;
long long g_batch_bytes = DEFAULT_BATCH_BYTES;
int g_fwd_variant = -1, g_bwd_variant = -1;   // -1: automatic

struct DevInfo {
    int sms = 0;
    int major = 0, minor = 0;
    int fwd_blocks[kNumFwd] = {};
    int bwd_blocks[kNumBwd] = {};
};
std::map<int, DevInfo> g_dev;

// Library-owned scratch of one (device, stream): control block, the two P1
// counter arrays (fixed capacity, so that a launch can clear the array of
// the next launch whatever its sizes), then the per-launch arrays.
struct Workspace {
    unsigned char *base = nullptr;
    size_t bytes = 0;
    int ctr_cap = 0;
};

size_t counters_end(int ctr_cap) { return 256 + ((size_t(8) * ctr_cap + 255) / 256) * 256; }
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
            auto setup = [&](const Variant &v, int *blocks) {
                const void *f = reinterpret_cast<const void *>(v.fn);
                if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v.smem()) !=
                        cudaSuccess ||
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, f, NTHREADS, v.smem()) != cudaSuccess)
                    return false;
                *blocks = std::max(*blocks, 1);
                return true;
            };
            bool ok = true;
            for (int i = 0; i < kNumFwd; ++i) ok = ok && setup(kFwdVariants[i], &d.fwd_blocks[i]);
            for (int i = 0; i < kNumBwd; ++i) ok = ok && setup(kBwdVariants[i], &d.bwd_blocks[i]);
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

// Returns the workspace of (device, stream) with room for `plan_bytes` of
// per-launch arrays and at least `ng` counters per array.
int ensure_workspace(int dev, cudaStream_t stream, size_t plan_bytes, int ng, unsigned char **out, int *ctr_cap) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace &w = g_ws[{dev, reinterpret_cast<uintptr_t>(stream)}];
    if (w.ctr_cap >= ng && w.bytes >= counters_end(w.ctr_cap) + plan_bytes) {
        *out = w.base;
        *ctr_cap = w.ctr_cap;
        return QS_OK;
    }
    int cap = std::max(w.ctr_cap, 4096);
    while (cap < ng) cap *= 2;
    const size_t need = counters_end(cap) + plan_bytes;
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
    w.ctr_cap = cap;
    *out = w.base;
    *ctr_cap = cap;
    return QS_OK;
}

// View of a [B,S,H,J,4] tensor for TMA boxes of `lt` lanes x `boxh` steps.
// lt <= 64: 3-D view [B][S][HJ*4 floats].  lt == 128 (HJ a multiple of 64):
// 4-D view [B][S][HJ/64][64*4 floats], boxes of two 64-lane blocks.  Boxes may
// reach past the tensor: TMA fills those cells with zeros on loads and skips
// them on stores.
int make_map(CUtensorMap *m, const float *ptr, int64_t B, int64_t S, int64_t HJ, int lt, int boxh) {
    if (lt == 128) {
        EncodeTiledFn fn = encode_fn();
        if (!fn) return QS_ERR_CUDA;
        cuuint64_t dims[4] = {256, (cuuint64_t)(HJ / 64), (cuuint64_t)S, (cuuint64_t)B};
        cuuint64_t strides[3] = {1024, (cuuint64_t)(HJ * 16), (cuuint64_t)(S * HJ * 16)};
        cuuint32_t box[4] = {256, 2, (cuuint32_t)boxh, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        return r == CUDA_SUCCESS ? QS_OK : QS_ERR_CUDA;
    }
    const int boxw = lt;
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

// Everything a launch needs, derived from the sizes alone (no device calls).
struct Plan {
    const Variant *v = nullptr;
    int vidx = 0;
    qs::Geometry geo{};
    qs::Schedule sch{};
    long long nitems = 0;
    size_t o_sc = 0, o_L = 0, o_W = 0, o_F = 0, o_H = 0, ws_bytes = 0;   // offsets past the counters
};

int pick_variant(bool bwd, int64_t HJ) {
    int forced;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        forced = bwd ? g_bwd_variant : g_fwd_variant;
    }
    const Variant *table = bwd ? kBwdVariants : kFwdVariants;
    const int count = bwd ? kNumBwd : kNumFwd;
    if (forced >= 0 && forced < count && (table[forced].lt != 128 || HJ % 64 == 0)) return forced;
    if (!bwd && HJ >= 128 && HJ % 64 == 0) return 0;
    if (HJ >= 64) return bwd ? 0 : 1;
    return bwd ? 1 : 2;
}


int make_plan(bool bwd, int64_t B, int64_t S, int64_t HJ, Plan *pl) {
    pl->vidx = pick_variant(bwd, HJ);
    if (pl->vidx < 0 || pl->vidx >= (bwd ? kNumBwd : kNumFwd)) return QS_ERR_DIMS;
    pl->v = bwd ? &kBwdVariants[pl->vidx] : &kFwdVariants[pl->vidx];
    const int LT = pl->v->lt, T = pl->v->T();
    qs::Geometry &g = pl->geo;
    g.S = S;
    g.HJ = (int)HJ;
    g.NGb = (int)((HJ + LT - 1) / LT);
    const long long NG = (long long)B * g.NGb;
    const long long C = (S + T - 1) / T;
    if (NG >= (1ll << 30) || C >= (1ll << 30)) return QS_ERR_DIMS;
    g.NG = (int)NG;
    g.C = (int)C;
    long long batch_bytes;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        batch_bytes = g_batch_bytes;
    }
    const long long in_per_group = (long long)LT * S * 16 * (bwd ? 2 : 1);
    long long gb = batch_bytes / std::max<long long>(in_per_group, 1);
    gb = std::max<long long>(1, std::min<long long>(gb, NG));
    pl->sch.GB = (int)gb;
    pl->sch.NB = (int)((NG + gb - 1) / gb);
    pl->sch.NSB = LT / 32;
    const long long slots = C * NG;
    pl->nitems = 2 * slots + NG * pl->sch.NSB;
    if (pl->nitems >= (1ll << 31) - (1 << 20)) return QS_ERR_DIMS;
    size_t off = 0;
    pl->o_sc = off;
    off = align_up(off + NG * pl->sch.NSB * 8, 256);
    const size_t per = (size_t)slots * LT * 16;
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
    pl->ws_bytes = off;
    return QS_OK;
}

int launch(bool bwd, const float *q, const float *d_cum, float *out, const float *init, float *d_init, int64_t B,
           int64_t S, int64_t HJ, cudaStream_t stream) {
    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;
    Plan pl;
    rc = make_plan(bwd, B, S, HJ, &pl);
    if (rc != QS_OK) return rc;
    unsigned char *ws = nullptr;
    int ctr_cap = 0;
    rc = ensure_workspace(dev, stream, pl.ws_bytes, pl.geo.NG, &ws, &ctr_cap);
    if (rc != QS_OK) return rc;
    unsigned char *data = ws + counters_end(ctr_cap);
    CUtensorMap qmap, dmap, omap;
    const int lt = pl.v->lt, T = pl.v->T();
    rc = make_map(&qmap, q, B, S, HJ, lt, T);
    if (rc == QS_OK) rc = make_map(&omap, out, B, S, HJ, lt, T);
    if (rc == QS_OK) rc = make_map(&dmap, bwd ? d_cum : q, B, S, HJ, lt, T);
    if (rc != QS_OK) return rc;
    qs::Arrays arr;
    arr.p1_count = reinterpret_cast<unsigned int *>(ws + 256);
    arr.sc_flags = reinterpret_cast<unsigned long long *>(data + pl.o_sc);
    arr.aggL = reinterpret_cast<float4 *>(data + pl.o_L);
    arr.carF = reinterpret_cast<float4 *>(data + pl.o_F);
    arr.aggW = bwd ? reinterpret_cast<float4 *>(data + pl.o_W) : nullptr;
    arr.carH = bwd ? reinterpret_cast<float4 *>(data + pl.o_H) : nullptr;
    qs::Control ctl;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ctl.timeout_ns = g_timeout_ns;
        ctl.stall_item = g_stall_item;
    }
    ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
    ctl.nitems = (int)pl.nitems;
    ctl.ctr_cap = ctr_cap;
    const int blocks = bwd ? di->bwd_blocks[pl.vidx] : di->fwd_blocks[pl.vidx];
    const int grid = (int)std::min<long long>(pl.nitems, (long long)di->sms * blocks);
    const float4 *init4 = reinterpret_cast<const float4 *>(init);
    float4 *dinit4 = reinterpret_cast<float4 *>(d_init);
    void *args[] = {&qmap, &dmap, &omap, (void *)&init4, (void *)&dinit4, &arr, &pl.geo, &pl.sch, &ctl};
    if (cudaLaunchKernel(reinterpret_cast<const void *>(pl.v->fn), dim3(grid), dim3(NTHREADS), args, pl.v->smem(),
                         stream) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
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
    g_batch_bytes = bytes > 0 ? (long long)bytes : DEFAULT_BATCH_BYTES;
    return QS_OK;
}

extern "C" int quat_cumprod_debug_set_variant(int fwd_variant, int bwd_variant) {
    if (fwd_variant >= kNumFwd || bwd_variant >= kNumBwd) return QS_ERR_DIMS;
    std::lock_guard<std::mutex> lk(g_mu);
    g_fwd_variant = fwd_variant < 0 ? -1 : fwd_variant;
    g_bwd_variant = bwd_variant < 0 ? -1 : bwd_variant;
    return QS_OK;
}

// Host-side check of the work-item schedule for these sizes (both
// directions): every P1 (chunk, group), SC (group, 32-lane block) and P3
// (chunk, group) item appears exactly once, and every item comes after the
// items it waits on (SC after all P1 items of its group, P3 after all SC
// items of its group).
extern "C" int quat_cumprod_debug_check_schedule(int64_t B, int64_t S, int64_t H, int64_t J) {
    const int dc = check_dims(B, S, H, J);
    if (dc == 1) return QS_OK;
    if (dc != QS_OK) return dc;
    for (int bwd = 0; bwd < 2; ++bwd) {
        Plan pl;
        const int rc = make_plan(bwd != 0, B, S, H * J, &pl);
        if (rc != QS_OK) return rc;
        const long long C = pl.geo.C, NG = pl.geo.NG;
        if (pl.nitems > (1ll << 26)) return QS_ERR_DIMS;   // keep the check cheap
        const long long NSB = pl.sch.NSB;
        std::vector<long long> p1(C * NG, -1), p3(C * NG, -1), sc(NG * NSB, -1);
        for (long long id = 0; id < pl.nitems; ++id) {
            const qs::Work w = qs::decode_item((int)id, pl.geo.NG, pl.geo.C, pl.sch);
            if (w.g < 0 || w.g >= NG) return -100;
            if (w.kind == qs::KIND_SC) {
                if (w.sb < 0 || w.sb >= NSB || sc[w.g * NSB + w.sb] != -1) return -101;
                sc[w.g * NSB + w.sb] = id;
                continue;
            }
            if (w.chunk < 0 || w.chunk >= C) return -102;
            std::vector<long long> &v = (w.kind == qs::KIND_P1) ? p1 : p3;
            long long &slot = v[(long long)w.chunk * NG + w.g];
            if (slot != -1) return -103;
            slot = id;
        }
        for (long long g = 0; g < NG; ++g) {
            long long first_sc = -1, last_sc = -1;
            for (long long k = 0; k < NSB; ++k) {
                const long long v = sc[g * NSB + k];
                if (v < 0) return -104;
                first_sc = (first_sc < 0 || v < first_sc) ? v : first_sc;
                last_sc = v > last_sc ? v : last_sc;
            }
            for (long long c = 0; c < C; ++c) {
                const long long a = p1[c * NG + g], z = p3[c * NG + g];
                if (a < 0 || z < 0) return -105;
                if (a > first_sc) return -106;
                if (last_sc > z) return -107;
            }
        }
    }
    return QS_OK;
}
