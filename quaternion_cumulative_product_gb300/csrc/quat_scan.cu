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
//  * Each call picks its design from the number of lane groups.
//    Walk (one kernel): one CTA per lane group streams the whole sequence
//    through a TMA ring and keeps the carries between chunks itself -- the
//    forward reads q once and writes cum once; the backward walks forward
//    over q for the carries, then backward over q and d_cum.
//    For too few lane groups to fill the GPU, the forward is the segmented
//    chained walk (one kernel, quat_segwalk.cuh): persistent CTAs take
//    (segment, lane group) units in order, walk a segment twice (the second
//    time from L2) and chain the segments by decoupled look-back.  The
//    backward, and the bf16 forward, use aggregate / carry / apply (three
//    kernels): every chunk is an independent tile --
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
#include "quat_chain.cuh"
#include "quat_segwalk.cuh"
#include "quat_segwalk_bwd.cuh"
#include "quat_segwalk_tab.cuh"
#include "quat_segwalk_ws.cuh"
#include "quat_short.cuh"
#include "quat_tiles.cuh"
#include "quat_walk.cuh"

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
    int threads() const { return lt * nseg + extra; }
    size_t smem() const { return smem_bytes; }
    bool chain = false;  // single-pass chained scan (forward): `agg` is the kernel
    // Backward walk: most CTAs in flight, per SM x 4 (0: one CTA per lane
    // group).  Fewer CTAs than groups walk the groups in equal waves.
    int cap_x4 = 0;
    // Segmented chained walk (forward): segments of `segk` chunks, persistent
    // CTAs; `agg` is the kernel (0: another design).
    int segk = 0;
    int extra = 0;   // threads besides the LT * NSEG compute threads (warp-specialised kernels)
    // Segmented walk whose look-back values carry their own state (reset for
    // the next launch by the kernel itself; see LbValues).
    bool sent = false;
    // Backward segmented walk: the carries-only forward pass it starts from
    // when it recomputes the carries.
    const Variant *pass = nullptr;
    // Forward segmented walk with per-unit tables (quat_segwalk_tab_fwd_kernel):
    // its own argument list.
    bool tab = false;
    // Short sequences (quat_short_*_kernel): the whole sequence of LT lanes in
    // one CTA of LT * nseg threads, n steps each; S <= smax (0: another design).
    int smax = 0;
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
#define QS_SEGWALK_FWD(LT, NSEG, N, NST, K)                                                         \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_fwd_kernel<qs::IoF32, LT, NSEG, N, NST, K>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_smem_bytes(LT, NSEG, N, NST), false, 0, K      \
    }
#define QS_SEGWALK_SENT_FWD(LT, NSEG, N, NST, K)                                                    \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_fwd_kernel<qs::IoF32, LT, NSEG, N, NST, K, true>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_smem_bytes(LT, NSEG, N, NST), false, 0, K, 0, true \
    }
#define QS_SEGWALK_WS_SENT_FWD(LT, NSEG, N, NST, K)                                                 \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_ws_fwd_kernel<qs::IoF32, LT, NSEG, N, NST, K, true>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_smem_bytes(LT, NSEG, N, NST), false, 0, K, 64, true \
    }
#define QS_SEGWALK_WS_FWD(LT, NSEG, N, NST, K)                                                      \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_ws_fwd_kernel<qs::IoF32, LT, NSEG, N, NST, K>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_smem_bytes(LT, NSEG, N, NST), false, 0, K, 64  \
    }
#define QS_SEGWALK_TAB_FWD(LT, NSEG, N, NST, K, NLB)                                                \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_tab_fwd_kernel<qs::IoF32, LT, NSEG, N, NST, K, NLB>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_tab_smem_bytes(LT, NSEG, N, NST, K), false, 0, K,    \
            32 + 32 * NLB, true, nullptr, true                                                      \
    }
#define QS_WALK_BWD(LT, NSEG, N, NSTF, NSTB, SELF)                                                  \
    Variant {                                                                                       \
        true, reinterpret_cast<const void *>(qs::quat_walk_bwd_kernel<qs::IoF32, LT, NSEG, N, NSTF, NSTB, SELF, false>), \
            nullptr, true, LT, NSEG, N, qs::walk_bwd_smem_bytes(LT, NSEG, N, NSTF, NSTB)            \
    }
#define QS_SHORT_FWD(LT, NS, R)                                                                     \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_short_fwd_kernel<qs::IoF32, LT, NS, R>), nullptr, false, LT, \
            NS, R, 0, false, 0, 0, 0, false, nullptr, false, NS * R                                 \
    }
#define QS_SHORT_BWD(LT, NS, R)                                                                     \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_short_bwd_kernel<qs::IoF32, LT, NS, R>), nullptr, true, LT, \
            NS, R, 0, false, 0, 0, 0, false, nullptr, false, NS * R                                 \
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
    QS_SEGWALK_FWD(32, 8, 8, 3, 4),      // 9: segmented chained walk, 32 lanes, segments of 4 x 64 steps
    QS_SEGWALK_WS_FWD(32, 8, 8, 4, 4),   // 10: the same, warp-specialised (producer and look-back warps)
    QS_SEGWALK_WS_FWD(16, 8, 8, 6, 4),   // 11: warp-specialised, 16 lanes, 6 x 16 KiB ring
    QS_SEGWALK_SENT_FWD(32, 8, 8, 3, 4),   // 12: as 9, one-latency look-back rounds (few lane groups)
    QS_SEGWALK_WS_SENT_FWD(32, 8, 8, 4, 4),   // 13: as 10, one-latency look-back rounds
    QS_SEGWALK_WS_SENT_FWD(16, 8, 8, 6, 4),   // 14: as 11, one-latency look-back rounds
    QS_SEGWALK_SENT_FWD(32, 8, 8, 3, 1),      // 15: as 12, segments of one chunk (short sequences)
    QS_SEGWALK_SENT_FWD(32, 8, 8, 3, 2),      // 16: as 12, segments of 2 chunks
    QS_SEGWALK_WS_SENT_FWD(16, 8, 8, 6, 1),   // 17: as 14, segments of one chunk
    QS_SEGWALK_WS_SENT_FWD(16, 8, 8, 6, 2),   // 18: as 14, segments of 2 chunks
    QS_SEGWALK_TAB_FWD(16, 8, 8, 3, 4, 1),    // 19: segmented walk with per-unit tables, no block barrier, 16 lanes
    QS_SEGWALK_TAB_FWD(16, 8, 8, 3, 4, 2),    // 20: as 19, two look-back warps
    QS_SEGWALK_TAB_FWD(32, 8, 8, 3, 4, 2),    // 21: as 20, 32 lanes
    QS_SEGWALK_TAB_FWD(16, 8, 8, 3, 2, 2),    // 22: as 20, segments of 2 chunks
    QS_SEGWALK_TAB_FWD(16, 8, 8, 3, 1, 2),    // 23: as 20, segments of one chunk
    QS_SEGWALK_TAB_FWD(32, 8, 8, 3, 2, 2),    // 24: as 22, 32 lanes
    QS_SHORT_FWD(4, 128, 8),                  // 25: short sequences (S <= 1024), 4 lanes a CTA
    QS_SHORT_FWD(2, 128, 8),                  // 26: as 25, 2 lanes
    QS_SHORT_FWD(8, 128, 8),                  // 27: as 25, 8 lanes (1024 threads)
    QS_SHORT_FWD(4, 256, 8),                  // 28: S <= 2048, 4 lanes (1024 threads)
    QS_SHORT_FWD(16, 32, 8),                  // 29: S <= 256, 16 lanes
};
#define QS_WALK_BWD_CAP(LT, NSEG, N, NSTF, NSTB, CAPX4)                                             \
    Variant {                                                                                       \
        true, reinterpret_cast<const void *>(qs::quat_walk_bwd_kernel<qs::IoF32, LT, NSEG, N, NSTF, NSTB, false, false>), \
            nullptr, true, LT, NSEG, N, qs::walk_bwd_smem_bytes(LT, NSEG, N, NSTF, NSTB), false, CAPX4 \
    }
// The carries-only forward pass of the segmented backward (its forward
// carries, one read of q): 16-lane groups, 4-stage ring; segments of 4 chunks
// and one look-back warp, or segments of 8 chunks and two look-back warps
// taking alternate units (fewer, longer look-backs).
const Variant kCarriesPassVariant = Variant{
    false, reinterpret_cast<const void *>(qs::quat_carries_pass_kernel<qs::IoF32, 16, 8, 8, 4, 4>), nullptr, false,
    16, 8, 8, qs::carries_pass_smem_bytes(16, 8, 8, 4, 4), false, 0, 4, 64, true};
const Variant kCarriesPassVariant2 = Variant{
    false, reinterpret_cast<const void *>(qs::quat_carries_pass_kernel<qs::IoF32, 16, 8, 8, 4, 8, 4, 2>), nullptr,
    false, 16, 8, 8, qs::carries_pass_smem_bytes(16, 8, 8, 4, 8), false, 0, 8, 96, true};
// The same for bfloat16 tensors (the carries stay fp32).
const Variant kCarriesPassVariantBf16 = Variant{
    false, reinterpret_cast<const void *>(qs::quat_carries_pass_kernel<qs::IoBF16, 16, 8, 8, 6, 4>), nullptr, false,
    16, 8, 8, qs::carries_pass_smem_bytes(16, 8, 8, 6, 4, 8), false, 0, 4, 64, true};
#define QS_SEGWALK_BWD(LT, NSEG, N, NST, K, MINB, LB, W2FWD)                                        \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_bwd_kernel<qs::IoF32, LT, NSEG, N, NST, K, MINB, LB, W2FWD>), \
            nullptr, true, LT, NSEG, N, qs::segwalk_bwd_smem_bytes(LT, NSEG, N, NST, K), false, 0, K, 64, true, \
            &kCarriesPassVariant                                                                    \
    }
#define QS_SEGWALK_BWD2(LT, NSEG, N, NST, K, MINB)                                                  \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_bwd_kernel<qs::IoF32, LT, NSEG, N, NST, K, MINB, 4, false, 2>), \
            nullptr, true, LT, NSEG, N, qs::segwalk_bwd_smem_bytes(LT, NSEG, N, NST, K), false, 0, K, 96, true, \
            &kCarriesPassVariant2                                                                   \
    }
#define QS_SEGWALK_BWD_LAG(LT, NSEG, N, NST, K, MINB, DL, LB)                                      \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_bwd_kernel<qs::IoF32, LT, NSEG, N, NST, K, MINB, LB, false, 2, DL>), \
            nullptr, true, LT, NSEG, N, qs::segwalk_bwd_smem_bytes(LT, NSEG, N, NST, K, 16, DL + 1), false, 0, K, 96, \
            true, &kCarriesPassVariant2                                                             \
    }
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
    QS_WALK_BWD_CAP(16, 8, 8, 4, 2, 8),   // 10: as 4, at most 2 CTAs per SM (more groups: equal waves)
    QS_SEGWALK_BWD(16, 8, 8, 2, 4, 2, 4, false),   // 11: segmented walk (few lane groups), 16 lanes, segments of 4 chunks, 2 x 32 KiB ring
    QS_SEGWALK_BWD(16, 8, 8, 3, 2, 2, 4, false),   // 12: as 11, segments of 2 chunks, 3 x 32 KiB ring
    QS_SEGWALK_BWD(32, 8, 8, 2, 4, 1, 4, false),   // 13: 32 lanes, 2 x 64 KiB ring (one CTA per SM)
    QS_SEGWALK_BWD(16, 8, 8, 2, 2, 2, 4, false),   // 14: as 11, segments of 2 chunks
    QS_SEGWALK_BWD(16, 8, 8, 2, 4, 2, 8, false),   // 15: as 11, look-back rounds of 8 predecessors
    QS_SEGWALK_BWD(16, 8, 8, 2, 4, 2, 2, false),   // 16: as 11, look-back rounds of 2 predecessors
    QS_SEGWALK_BWD(16, 8, 8, 3, 2, 2, 8, false),   // 17: as 12, look-back rounds of 8 predecessors
    QS_SEGWALK_BWD(16, 8, 8, 2, 4, 2, 4, true),    // 18: as 11, walk 2 left to right
    QS_SEGWALK_BWD(16, 8, 8, 3, 2, 2, 4, true),    // 19: as 12, walk 2 left to right
    QS_SEGWALK_BWD(16, 8, 8, 2, 3, 2, 4, true),    // 20: segments of 3 chunks, walk 2 left to right
    QS_SEGWALK_BWD(16, 8, 8, 2, 1, 2, 4, false),   // 21: as 11, segments of one chunk (short sequences)
    QS_SEGWALK_BWD2(16, 8, 8, 2, 4, 2),            // 22: as 11, two look-back warps (alternate units; so is its carries pass)
    QS_SEGWALK_BWD2(16, 8, 8, 2, 2, 2),            // 23: as 14, two look-back warps
    QS_SEGWALK_BWD2(16, 8, 8, 3, 2, 2),            // 24: as 12, two look-back warps
    QS_SHORT_BWD(4, 128, 8),                       // 25: short sequences (S <= 1024), 4 lanes a CTA
    QS_SHORT_BWD(2, 128, 8),                       // 26: as 25, 2 lanes
    QS_SHORT_BWD(8, 64, 8),                        // 27: S <= 512, 8 lanes
    QS_SHORT_BWD(2, 256, 8),                       // 28: S <= 2048, 2 lanes
    QS_SHORT_BWD(16, 32, 8),                       // 29: S <= 256, 16 lanes
    QS_SEGWALK_BWD_LAG(16, 8, 8, 2, 2, 2, 3, 4),   // 30: as 23, walk 2 three units behind walk 1
    QS_SEGWALK_BWD_LAG(16, 8, 8, 2, 2, 2, 2, 4),   // 31: as 23, walk 2 two units behind
    QS_SEGWALK_BWD_LAG(16, 8, 8, 2, 3, 2, 2, 4),   // 32: as 31, segments of 3 chunks
    QS_SEGWALK_BWD_LAG(16, 8, 8, 2, 2, 2, 2, 8),   // 33: as 31, look-back batches of 8
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
#define QS_WALK_BWD16_MINB(LT, NSEG, N, NSTF, NSTB, MINB)                                           \
    Variant {                                                                                       \
        true,                                                                                       \
            reinterpret_cast<const void *>(                                                         \
                qs::quat_walk_bwd_kernel<qs::IoBF16, LT, NSEG, N, NSTF, NSTB, false, false, MINB>), \
            nullptr, true, LT, NSEG, N, qs::walk_bwd_smem_bytes(LT, NSEG, N, NSTF, NSTB, 8)         \
    }
#define QS_VARIANT16(B, LT, N)                                                                      \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_agg_kernel<qs::IoBF16, B, LT, N>),           \
            reinterpret_cast<const void *>(qs::quat_apply_kernel<qs::IoBF16, B, LT, N>), B, LT,     \
            NTHREADS / (LT), N, qs::tile_smem_bytes(B, LT, N, 8)                                    \
    }
#define QS_SEGWALK_WS_SENT_FWD16(LT, NSEG, N, NST, K)                                               \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_ws_fwd_kernel<qs::IoBF16, LT, NSEG, N, NST, K, true>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_smem_bytes(LT, NSEG, N, NST, 8), false, 0, K, 64, true \
    }
#define QS_SEGWALK_BWD16(LT, NSEG, N, NST, K, MINB)                                                 \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_bwd_kernel<qs::IoBF16, LT, NSEG, N, NST, K, MINB, 4, false>), \
            nullptr, true, LT, NSEG, N, qs::segwalk_bwd_smem_bytes(LT, NSEG, N, NST, K, 8), false, 0, K, 64, true, \
            &kCarriesPassVariantBf16                                                                \
    }
#define QS_SEGWALK_TAB_FWD16(LT, NSEG, N, NST, K, NLB)                                              \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_tab_fwd_kernel<qs::IoBF16, LT, NSEG, N, NST, K, NLB>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_tab_smem_bytes(LT, NSEG, N, NST, K, 8), false, 0, K, \
            32 + 32 * NLB, true, nullptr, true                                                      \
    }
#define QS_SEGWALK_SENT_FWD16(LT, NSEG, N, NST, K)                                                  \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_fwd_kernel<qs::IoBF16, LT, NSEG, N, NST, K, true>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_smem_bytes(LT, NSEG, N, NST, 8), false, 0, K, 0, true \
    }
#define QS_SEGWALK_FWD16(LT, NSEG, N, NST, K)                                                       \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_segwalk_fwd_kernel<qs::IoBF16, LT, NSEG, N, NST, K>), \
            nullptr, false, LT, NSEG, N, qs::segwalk_smem_bytes(LT, NSEG, N, NST, 8), false, 0, K   \
    }
#define QS_SHORT_FWD16(LT, NS, R)                                                                   \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_short_fwd_kernel<qs::IoBF16, LT, NS, R>), nullptr, false, LT, \
            NS, R, 0, false, 0, 0, 0, false, nullptr, false, NS * R                                 \
    }
#define QS_SHORT_BWD16(LT, NS, R)                                                                   \
    Variant {                                                                                       \
        false, reinterpret_cast<const void *>(qs::quat_short_bwd_kernel<qs::IoBF16, LT, NS, R>), nullptr, true, LT, \
            NS, R, 0, false, 0, 0, 0, false, nullptr, false, NS * R                                 \
    }
const Variant kFwdBf16Variants[] = {
    QS_WALK_FWD16(32, 8, 8, 6),            // 0: 32 lanes x 64 steps, 6 x 16 KiB ring
    QS_WALK_FWD16(16, 8, 8, 6),            // 1: 16 lanes x 64 steps (128 threads), 6 x 8 KiB
    QS_WALK_FWD16(16, 16, 8, 4),           // 2: 16 lanes x 128 steps (256 threads), 4 x 16 KiB
    QS_WALK_FWD16(32, 16, 4, 6),           // 3: 32 lanes x 64 steps (512 threads), 6 x 16 KiB
    QS_VARIANT16(false, 32, 8),            // 4: three kernels, 64-step chunks
    QS_SEGWALK_FWD16(32, 8, 8, 3, 4),      // 5: segmented chained walk (few lane groups)
    QS_SEGWALK_SENT_FWD16(32, 8, 8, 3, 4), // 6: as 5, one-latency look-back rounds
    QS_SEGWALK_WS_SENT_FWD16(16, 8, 8, 6, 4),   // 7: segmented walk, warp-specialised, 16 lanes
    QS_SHORT_FWD16(2, 128, 8),             // 8: short sequences (S <= 1024), 2 lanes a CTA
    QS_SHORT_FWD16(4, 256, 8),             // 9: S <= 2048, 4 lanes (1024 threads)
    QS_SEGWALK_TAB_FWD16(32, 8, 8, 3, 2, 2),   // 10: segmented walk with per-unit tables, 32 lanes
};
const Variant kBwdBf16Variants[] = {
    QS_WALK_BWD16(16, 8, 8, 8, 4, false),  // 0: 16 lanes x 64 steps (128 threads), 64 KiB rings
    QS_WALK_BWD16(16, 8, 8, 8, 4, true),   // 1: the same, each thread folds its own carries
    QS_WALK_BWD16(16, 16, 4, 8, 4, false), // 2: 16 lanes x 64 steps (256 threads), 64 KiB rings
    QS_WALK_BWD16(32, 8, 8, 8, 4, false),  // 3: 32 lanes x 64 steps (256 threads), 128 KiB rings
    QS_VARIANT16(true, 32, 8),             // 4: three kernels, 64-step chunks (few lane groups)
    QS_WALK_BWD16_MINB(16, 8, 8, 8, 4, 3), // 5: as 0, registers capped for 3 CTAs per SM (many lane groups)
    QS_SEGWALK_BWD16(16, 8, 8, 3, 4, 2),   // 6: segmented walk (after the carries pass), segments of 4 chunks
    QS_SEGWALK_BWD16(16, 8, 8, 3, 2, 2),   // 7: segmented walk, segments of 2 chunks
    QS_SHORT_BWD16(2, 128, 8),             // 8: short sequences (S <= 1024), 2 lanes a CTA
    QS_SHORT_BWD16(8, 64, 8),              // 9: S <= 512, 8 lanes
    QS_SHORT_BWD16(2, 256, 8),             // 10: S <= 2048, 2 lanes
};
#undef QS_VARIANT16
#undef QS_SHORT_FWD16
#undef QS_SHORT_BWD16
#undef QS_SEGWALK_FWD16
#undef QS_SEGWALK_SENT_FWD16
#undef QS_SEGWALK_TAB_FWD16
#undef QS_SEGWALK_WS_SENT_FWD16
#undef QS_SEGWALK_BWD16
#undef QS_WALK_FWD16
#undef QS_WALK_BWD16
#undef QS_WALK_BWD16_MINB
constexpr int kNumFwdBf16 = sizeof(kFwdBf16Variants) / sizeof(kFwdBf16Variants[0]);
constexpr int kFwdBf16Default = 1, kBwdBf16Default = 0;   // walks
// The bf16 forward walk only from three lane groups of 16 per SM: with half
// the bytes a walk's time is its own latency, which only many CTAs per SM hide
// (16 x 8192 x 32 x 32, 1024 groups: walk 0.86 of the copy bandwidth at 16
// bytes per element, against 0.72).  With fewer, the segmented walk with
// per-unit tables and 32-lane groups (8 x 4096 x 16 x 32: 0.61 against the
// walk's 0.53; 1 x 131072 x 16 x 16: 0.61 against 0.49 for the segmented walk
// with status words; 2 x 65536 x 32 x 32: 0.71 against 0.56).
constexpr int kFwdBf16Few = 10, kBwdBf16Few = 4;
constexpr int kFwdBf16WalkGroupsPerSm = 3;
constexpr int kFwdBf16Three = 4;   // the aggregate / carry / apply forward
constexpr int kBwdBf16Three = 4;   // the aggregate / carry / apply backward
// The bf16 backward walk with more lane groups than two CTAs per SM hold: its
// registers capped so that three fit (168 instead of 205 a thread).  On
// 16 x 8192 x 32 x 32 (1024 groups) it measured 0.528 against 0.497 of the copy
// bandwidth; on 8 x 4096 x 16 x 32 (256 groups) 0.401 against 0.418.
constexpr int kBwdBf16Many = 5;
constexpr int kNumBwdBf16 = sizeof(kBwdBf16Variants) / sizeof(kBwdBf16Variants[0]);
#undef QS_VARIANT
#undef QS_SEGWALK_FWD
#undef QS_SEGWALK_WS_FWD
#undef QS_SEGWALK_SENT_FWD
#undef QS_SEGWALK_WS_SENT_FWD
#undef QS_SEGWALK_TAB_FWD
#undef QS_WALK_FWD
#undef QS_WALK_BWD
#undef QS_WALK_BWD_CAP
#undef QS_SEGWALK_BWD
#undef QS_SEGWALK_BWD2
#undef QS_SEGWALK_BWD_LAG
#undef QS_SHORT_FWD
#undef QS_SHORT_BWD
// Lanes per block of the carry scan (sequences of more than 256 chunks).
constexpr int kCarryScanLanes = 2;

// Automatic choice between the two designs.  A walk keeps one CTA per lane
// group for the whole sequence, so it needs enough lane groups to keep every
// SM streaming (measured: 128 groups of 32 lanes forward and 256 groups of 16
// lanes backward already beat the three-kernel path on 152 SMs).  With fewer
// lanes -- long sequences of few lanes -- the three-kernel path, which splits
// the sequence into independent tiles, is the faster one (forward: the
// segmented chained walk, which also cuts the sequence).  The backward walk
// runs at most two CTAs per SM: with more lane groups than that (16 x 8192 x
// 32 x 32: 1024 groups) each CTA walks several in equal waves, measured 5%
// faster than one CTA per group in the hardware's own waves.
constexpr int kWalkFwd = 4, kWalkBwd = 10, kThreeFwd = 0, kThreeBwd = 0;
// Backward with too few lane groups for a walk: the segmented walk (after a
// carries-only forward pass when the carries are not saved: 64 bytes per
// element of DRAM instead of the three kernels' 80), see pick_variant.
constexpr int kSegBwdLag = 31;   // segments of 2 chunks, walk 2 two units behind walk 1
// Forward with too few lane groups for a walk: the segmented walk with
// per-unit tables and two look-back warps (no block barrier), segments of 2
// chunks; 32-lane groups when there are at most 32 of them.  Measured alone
// (fraction of the copy bandwidth at 32 bytes per element) against the
// warp-specialised segmented walk with per-chunk folds (configuration 14):
// 1 x 131072 x 16 x 16 0.93 (configuration 24) / 0.90 (22) against 0.77;
// 2 x 65536 x 32 x 32 0.98 (22) / 0.97 (24) against 0.83; 2 x 4096 x 16 x 32
// 0.68 (24) / 0.63 (22) against 0.49; 4 x 1024 x 8 x 16 0.17 for both against
// 0.15.  (On 8 x 4096 x 16 x 32 the walk stays ahead: 0.94 against 0.91.)
constexpr int kSegFwd = 22, kSegFwdFew = 24;
constexpr long long kSegFwdFewGroups = 32;   // lane groups of 32
constexpr int kNumFwd = sizeof(kFwdVariants) / sizeof(kFwdVariants[0]);
constexpr int kNumBwd = sizeof(kBwdVariants) / sizeof(kBwdVariants[0]);

std::mutex g_mu;
unsigned long long g_timeout_ns = DEFAULT_TIMEOUT_NS;
int g_stall_tile = -1;
int g_fwd_variant = -1, g_bwd_variant = -1;   // -1: automatic
int g_fwd_variant16 = -1, g_bwd_variant16 = -1;
int g_bwd_cap = -1;   // CTAs in flight of the backward walk (-1: the variant's)

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
// Device -> address of quat_cumprod_bwd_noalloc's fixed scratch array (set up
// by that call's first use on the device).
std::map<int, unsigned char *> g_noalloc_ptr;
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
            setup(kCarriesPassVariant);
            setup(kCarriesPassVariant2);
            setup(kCarriesPassVariantBf16);
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

// Head of the status-word allocation: the counters of the segmented chained
// walk (tickets taken, CTAs finished, units done), padded; status words start
// after it.
constexpr size_t kFlagsHead = 256;

// Look-back values of the segmented walks that carry their own state (Variant
// `sent`): per (device, stream, kind of launch) an allocation no other kernel
// writes, holding two sets of `narr` buffers of `n` entries each (forward:
// segment products and inclusive values; backward: the maps' V and A and the
// inclusive values).  A launch reads the set `next` and resets the other one
// for the launch after it; the host clears both when the entry layout changes
// (and when the allocation is new, or a launch failed to be enqueued).  Each
// kind keeps its own buffers, so that alternating launches of different kinds
// on a stream (a forward, a backward and its carries pass) need no clearing.
enum LbKind { LB_FWD = 0, LB_CARRIES = 1, LB_BWD = 2 };
constexpr int kLbMaxArrays = 3;
struct LbValues {
    unsigned char *base = nullptr;
    size_t bytes = 0;
    long long n = -1;   // entries per buffer of the layout the buffers are clean for; -1: none
    int next = 0;       // the set the next launch reads
};
struct LbKey {
    int dev;
    uintptr_t stream;
    int kind;
    bool operator<(const LbKey &o) const {
        return dev != o.dev ? dev < o.dev : stream != o.stream ? stream < o.stream : kind < o.kind;
    }
};
std::map<LbKey, LbValues> g_lbv;
// Held from choosing a launch's set to enqueueing it, so that launches on a
// stream are enqueued in the order their sets were handed out.
std::mutex g_lbv_launch_mu;

// The `narr` buffers a launch of `n` entries per buffer reads (cur) and the
// ones it resets (next); enqueues the clearing memset if needed.
int lb_values(int dev, cudaStream_t stream, int kind, long long n, int narr, float4 **cur, float4 **next) {
    std::lock_guard<std::mutex> lk(g_mu);
    LbValues &w = g_lbv[{dev, reinterpret_cast<uintptr_t>(stream), kind}];
    const size_t arr = align_up((size_t)n * 16, 256), need = 2 * (size_t)narr * arr;
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
        w.base = static_cast<unsigned char *>(p);
        w.bytes = bytes;
        w.n = -1;
    }
    if (w.n != n) {
        if (cudaMemsetAsync(w.base, 0xff, need, stream) != cudaSuccess) {
            cudaGetLastError();
            w.n = -1;
            return QS_ERR_CUDA;
        }
        w.n = n;
        w.next = 0;
    }
    const int b = w.next;
    for (int i = 0; i < narr; ++i) {
        cur[i] = reinterpret_cast<float4 *>(w.base + (size_t)(b * narr + i) * arr);
        next[i] = reinterpret_cast<float4 *>(w.base + (size_t)((b ^ 1) * narr + i) * arr);
    }
    w.next = b ^ 1;
    return QS_OK;
}

// After a launch that was not enqueued: the next one starts from cleared buffers.
void lb_values_invalidate(int dev, cudaStream_t stream, int kind) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_lbv[{dev, reinterpret_cast<uintptr_t>(stream), kind}].n = -1;
}

// CTAs of a persistent kernel: as many as are resident at once on the device
// (per (device, kernel), computed once).
std::map<std::pair<int, const void *>, int> g_occ;
int persistent_grid(int dev, const Variant *v, int *grid) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occ.find({dev, v->agg});
    if (it == g_occ.end()) {
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, v->agg, v->threads(), v->smem()) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        it = g_occ.emplace(std::make_pair(dev, v->agg), per_sm * sms).first;
    }
    *grid = it->second;
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
    int walk_grid = 0;   // CTAs of a walk kernel
    size_t o_L = 0, o_W = 0, o_F = 0, o_H = 0, o_I = 0, ws_bytes = 0;
};

int layout_plan(bool bwd, int64_t B, int64_t S, int64_t HJ, int sms, Plan *pl, Mode mode);

// The backward for few lane groups (LT = 16 groups, C 64-step chunks), both
// measured on one GB300 with L2 flushed before every call (fraction of the
// copy bandwidth at 48 bytes per element), the segmented walk with two
// look-back warps:
//  * on long sequences of few groups (at least 4 units of 4 chunks per SM),
//    segments of 2 chunks with walk 2 two units behind walk 1, so that a
//    unit's look-back (about 3 us, running deep) ends before its second walk
//    is due: from saved carries 1 x 131072 x 16 x 16 0.79 (0.75 with segments
//    of 4 chunks and walk 2 one unit behind, 0.58 with 2 chunks one unit
//    behind), 1 x 262144 x 16 x 16 0.80, 2 x 65536 x 16 x 16 0.78; recomputing
//    the carries (the carries pass first) 0.61 / 0.63 / 0.61 against 0.58 /
//    0.60 / 0.58 for the three kernels;
//  * with 64 groups or more, segments of 2 chunks one unit behind, one CTA
//    per SM (2 x 65536 x 32 x 32: 0.92 from saved carries, 0.71 recomputing
//    against 0.60 for the three kernels; 4 x 32768 x 16 x 16: 0.80 / 0.62);
//  * with few units, from saved carries the same (4 x 4096 x 8 x 16), and
//    recomputing the three kernels.
constexpr int kSegBwdShort = 24;           // segments of 2 chunks, two look-back warps, one CTA per SM
constexpr long long kSegBwdManyGroups = 64;

// Short sequences with too few lane groups for a walk: the whole sequence of
// a few lanes in one CTA (no look-back, one launch), the configuration that
// fits S with the fewest idle segments.  Measured alone on 152 SMs (L2
// flushed; a trivial kernel timed the same way takes 6.8 us):
//   4 x 1024 x 8 x 16: forward 10.9 us against 15.0 (segmented walk),
//                      backward 12.9 us against 23.2 (three kernels);
//   2 x 2048 x 16 x 16: forward 12.9 against 17.0, backward 23.2 against 31.4;
//   4 x 512 x 16 x 16: backward 12.9 (8 lanes, S <= 512) against 17.0 (2 or 4
//                      lanes) and 31.4 (segmented walk).
// (4 steps a thread instead of 8, with twice the segments: slower, 19.1 us
// against 13.0 for the backward of 4 x 1024 x 8 x 16.)
// Returns the configuration in the fp32 or bf16 table, or -1 past 2048 steps.
int short_variant(bool bwd, int64_t S, bool bf16) {
    if (S > 2048) return -1;
    if (bf16) {
        if (bwd) return S <= 512 ? 9 : S <= 1024 ? 8 : 10;
        return S <= 1024 ? 8 : 9;
    }
    if (bwd) return S <= 512 ? 27 : S <= 1024 ? 25 : 28;
    return S <= 1024 ? 26 : 28;
}

int pick_variant(bool bwd, int64_t B, int64_t S, int64_t HJ, int sms, Mode mode) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const int forced = bwd ? g_bwd_variant : g_fwd_variant;
        // (a short-sequence configuration only where the sequence fits it)
        if (forced >= 0 && (S <= (bwd ? kBwdVariants : kFwdVariants)[forced].smax ||
                            (bwd ? kBwdVariants : kFwdVariants)[forced].smax == 0))
            return forced;
    }
    const Variant &w = bwd ? kBwdVariants[kWalkBwd] : kFwdVariants[kWalkFwd];
    const long long groups = (long long)B * ((HJ + w.lt - 1) / w.lt);
    const long long need = bwd ? 3ll * sms / 2 : 3ll * sms / 4;
    if (groups >= need) return bwd ? kWalkBwd : kWalkFwd;
    const int sv = short_variant(bwd, S, false);
    if (sv >= 0) return sv;
    if (bwd) {
        const long long units4 = groups * ((S + 4 * 64 - 1) / (4 * 64));   // segments of 4 chunks
        if (groups >= kSegBwdManyGroups) return kSegBwdShort;
        if (units4 >= 4ll * sms) return kSegBwdLag;
        return mode == Mode::FROM_CARRIES ? kSegBwdShort : kThreeBwd;
    }
    return groups <= kSegFwdFewGroups ? kSegFwdFew : kSegFwd;
}

// `capturing`: the call is being captured into a CUDA graph, whose launches
// are replayed with the same arguments.  The segmented walk and the chained
// scan keep state from one launch to the next (the epoch of their status
// words, or which buffers of self-describing values a launch reads), so a
// replay would take the previous replay's values for published ones; under
// capture the forward therefore uses the aggregate / carry / apply kernels,
// which keep none.  Eager plans of those designs reserve the workspace of that
// forward as well, so a call before the capture sizes it.
int make_plan(bool bwd, int64_t B, int64_t S, int64_t HJ, int sms, Plan *pl, Mode mode = Mode::PLAIN,
              bool bf16 = false, bool capturing = false) {
    int vi = 0;
    if (bf16) {
        int forced;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            forced = bwd ? g_bwd_variant16 : g_fwd_variant16;
        }
        const Variant *fv = forced < 0 ? nullptr : bwd ? &kBwdBf16Variants[forced] : &kFwdBf16Variants[forced];
        if (fv != nullptr && (fv->smax == 0 || S <= fv->smax)) {
            vi = forced;
        } else {   // the same rule as for fp32: a walk when the lane groups fill the GPU
            const int wi = bwd ? kBwdBf16Default : kFwdBf16Default;
            const Variant &w = bwd ? kBwdBf16Variants[wi] : kFwdBf16Variants[wi];
            const long long groups = (long long)B * ((HJ + w.lt - 1) / w.lt);
            const long long need = bwd ? 3ll * sms / 2 : (long long)kFwdBf16WalkGroupsPerSm * sms;
            vi = groups >= need ? wi : (bwd ? kBwdBf16Few : kFwdBf16Few);
            if (groups < need && short_variant(bwd, S, true) >= 0) vi = short_variant(bwd, S, true);
            if (bwd && groups > 2ll * sms) vi = kBwdBf16Many;
        }
    } else {
        vi = pick_variant(bwd, B, S, HJ, sms, mode);
    }
    const Variant *v = bf16 ? (bwd ? &kBwdBf16Variants[vi] : &kFwdBf16Variants[vi])
                            : bwd ? &kBwdVariants[vi] : &kFwdVariants[vi];
    if (mode != Mode::PLAIN && v->chain) {   // the chained scan writes no carries: take the three kernels
        vi = kThreeFwd;
        v = &kFwdVariants[vi];
    }
    if (mode != Mode::PLAIN && v->T() != QS_CARRY_STEPS && v->smax == 0) {
        // The carries are defined on QS_CARRY_STEPS-step chunks: keep the
        // design, take its default configuration (which has that chunk).
        vi = v->walk ? (bwd ? kWalkBwd : kWalkFwd) : (bwd ? kThreeBwd : kThreeFwd);
        v = bwd ? &kBwdVariants[vi] : &kFwdVariants[vi];
    }
    if (mode == Mode::FROM_CARRIES && v->walk) v = &kBwdGiven;
    const bool stateful = v->chain || v->segk > 0;
    const int vthree = bf16 ? (bwd ? kBwdBf16Three : kFwdBf16Three) : (bwd ? kThreeBwd : kThreeFwd);
    const Variant *three = bf16 ? (bwd ? &kBwdBf16Variants[vthree] : &kFwdBf16Variants[vthree])
                                : (bwd ? &kBwdVariants[vthree] : &kFwdVariants[vthree]);
    if (capturing && stateful) {
        vi = vthree;
        v = three;
    }
    pl->vi = vi;
    pl->v = v;
    int rc = layout_plan(bwd, B, S, HJ, sms, pl, mode);
    if (rc != QS_OK || capturing || !stateful) return rc;
    Plan p3;
    p3.vi = vthree;
    p3.v = three;
    rc = layout_plan(bwd, B, S, HJ, sms, &p3, mode);
    if (rc == QS_OK && p3.ws_bytes > pl->ws_bytes) pl->ws_bytes = p3.ws_bytes;
    return rc;
}

// Geometry and workspace layout of the configuration pl->v.
int layout_plan(bool bwd, int64_t B, int64_t S, int64_t HJ, int sms, Plan *pl, Mode mode) {
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
    if (pl->v->smax > 0) {   // short sequences: one CTA per lane group, nothing but the status block
        pl->ws_bytes = off;
        return QS_OK;
    }
    if (pl->v->segk > 0 && bwd) {
        // Backward segmented walk: the look-back values live apart (LbValues),
        // the ticket counters in the head of the status-word allocation; the
        // workspace holds the carries of the carries-only pass, [B, C, H*J].
        pl->o_L = kFlagsHead;
        if (mode != Mode::FROM_CARRIES) {
            pl->o_F = off;
            off = align_up(off + (size_t)B * C * HJ * 16, 256);
        }
        pl->ws_bytes = off;
        return QS_OK;
    }
    if (pl->v->segk > 0) {
        // Segmented chained walk: per unit (segment, lane group) and lane the
        // segment product and the inclusive value; the status words and the
        // ticket counter live apart (see chain_flags).
        const long long units = NG * ((C + pl->v->segk - 1) / pl->v->segk);
        const size_t pu = (size_t)units * LT * 16;
        pl->o_L = kFlagsHead + (size_t)units * LT * 4;
        pl->o_W = off;   // segment products
        off = align_up(off + pu, 256);
        pl->o_F = off;   // inclusive values
        off = align_up(off + pu, 256);
        pl->ws_bytes = off;
        return QS_OK;
    }
    if (pl->v->chain) {
        // Chained scan: status block, then per tile and lane the chunk product
        // and the inclusive value (the status words live apart, see chain_flags).
        pl->o_L = kFlagsHead + (size_t)pl->tiles * LT * 4;   // bytes of status words (their own allocation)
        pl->o_W = off;   // chunk products
        off = align_up(off + per, 256);
        pl->o_F = off;   // inclusive values
        off = align_up(off + per, 256);
        pl->ws_bytes = off;
        return QS_OK;
    }
    if (pl->v->walk) {
        // One CTA per lane group, or (backward, capped) equal waves of groups.
        long long cap = NG;
        if (bwd) {
            int forced;
            {
                std::lock_guard<std::mutex> lk(g_mu);
                forced = g_bwd_cap;
            }
            if (forced > 0) cap = forced;
            else if (pl->v->cap_x4 > 0) cap = std::max(1ll, (long long)pl->v->cap_x4 * sms / 4);
        }
        const long long waves = (NG + cap - 1) / cap;
        pl->walk_grid = (int)((NG + waves - 1) / waves);
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

// The control block of a launch: the wait limit, the test hook's stalled tile
// (`stall`: this launch is the first kernel of its call) and the status block.
qs::Control control_block(unsigned char *ws, bool stall) {
    qs::Control ctl;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ctl.timeout_ns = g_timeout_ns;
        ctl.stall_tile = stall ? g_stall_tile : -1;
    }
    ctl.hdr = reinterpret_cast<qs::WsHeader *>(ws);
    return ctl;
}

// Geometry of LT-lane groups and T-step chunks.
qs::Geometry geometry(int64_t B, int64_t S, int64_t HJ, int LT, int T) {
    qs::Geometry g;
    g.S = S;
    g.HJ = (int)HJ;
    g.NGb = (int)((HJ + LT - 1) / LT);
    g.NG = (int)(B * g.NGb);
    g.C = (int)((S + T - 1) / T);
    g.NL = g.NG * LT;
    return g;
}

// The backward segmented walk (pl.v): without saved carries, first the
// carries-only forward pass writes every chunk's carry into the workspace.
// Both launches are enqueued under the look-back buffers' ordering lock.
int launch_segwalk_bwd(const Plan &pl, int dev, unsigned char *ws, const void *q, const void *d_cum, void *d_q,
                       const void *init, void *d_init, int64_t B, int64_t S, int64_t HJ, cudaStream_t stream,
                       Mode mode, float *carries, bool bf16) {
    const Variant *v = pl.v;
    const int eb = bf16 ? 8 : 16;
    uint32_t epoch = 0, *flags = nullptr;
    int rc = chain_flags(dev, stream, pl.o_L, &flags, &epoch);
    if (rc != QS_OK) return rc;
    unsigned int *tickets = flags;   // counters, zero between launches (shared: launches on a stream are ordered)
    std::lock_guard<std::mutex> order(g_lbv_launch_mu);
    const float4 *car = reinterpret_cast<const float4 *>(carries);
    const bool pass = mode != Mode::FROM_CARRIES;
    if (pass) {
        const Variant &pv = *v->pass;
        qs::Geometry pg = geometry(B, S, HJ, pv.lt, pv.T());
        CUtensorMap pmap;
        rc = make_map(&pmap, q, B, S, HJ, pv.lt, pv.T(), eb);
        if (rc != QS_OK) return rc;
        int grid = 0;
        rc = persistent_grid(dev, &pv, &grid);
        if (rc != QS_OK) return rc;
        const long long units = (long long)pg.NG * ((pg.C + pv.segk - 1) / pv.segk);
        if (grid > units) grid = (int)units;
        float4 *cur[kLbMaxArrays], *nxt[kLbMaxArrays];
        rc = lb_values(dev, stream, LB_CARRIES, units * pv.lt, 2, cur, nxt);
        if (rc != QS_OK) return rc;
        qs::Control ctl = control_block(ws, true);
        float4 *carw = reinterpret_cast<float4 *>(ws + pl.o_F);
        const void *init4 = init;
        void *args[] = {&pmap, &init4, &carw, &tickets, &cur[0], &cur[1], &nxt[0], &nxt[1], &pg, &ctl};
        if (cudaLaunchKernel(pv.agg, dim3((unsigned)grid), dim3(pv.threads()), args, pv.smem(), stream) !=
            cudaSuccess) {
            cudaGetLastError();
            lb_values_invalidate(dev, stream, LB_CARRIES);
            return QS_ERR_CUDA;
        }
        car = carw;
    }
    CUtensorMap qmap, dmap;
    rc = make_map(&qmap, q, B, S, HJ, v->lt, v->T(), eb);
    if (rc == QS_OK) rc = make_map(&dmap, d_cum, B, S, HJ, v->lt, v->T(), eb);
    if (rc != QS_OK) return rc;
    int grid = 0;
    rc = persistent_grid(dev, v, &grid);
    if (rc != QS_OK) return rc;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_bwd_cap > 0 && grid > g_bwd_cap) grid = g_bwd_cap;   // test hook: fewer CTAs in flight
    }
    const long long units = (long long)pl.geo.NG * ((pl.geo.C + v->segk - 1) / v->segk);
    if (grid > units) grid = (int)units;
    float4 *cur[kLbMaxArrays], *nxt[kLbMaxArrays];
    rc = lb_values(dev, stream, LB_BWD, units * v->lt, 3, cur, nxt);
    if (rc != QS_OK) return rc;
    qs::Control ctl = control_block(ws, !pass);
    qs::Geometry geo = pl.geo;
    void *dq4 = d_q, *dinit4 = d_init;
    void *args[] = {&qmap, &dmap, &car, &dq4, &dinit4, &tickets, &cur[0], &cur[1], &cur[2], &nxt[0], &nxt[1],
                    &nxt[2], &geo, &ctl};
    if (cudaLaunchKernel(v->agg, dim3((unsigned)grid), dim3(v->threads()), args, v->smem(), stream) != cudaSuccess) {
        cudaGetLastError();
        lb_values_invalidate(dev, stream, LB_BWD);
        return QS_ERR_CUDA;
    }
    return QS_OK;
}

// Short sequences (pl.v->smax > 0): one launch, one CTA per lane group.  From
// saved carries the backward takes init = carries[:, 0] and recomputes the rest
// (the whole sequence is in the CTA's registers anyway).
int launch_short(const Plan &pl, bool bwd, const void *q, const void *d_cum, void *out, const void *init,
                 void *d_init, int64_t S, int64_t HJ, cudaStream_t stream, Mode mode, float *carries, bool bf16) {
    const void *init_p = init;
    long long init_stride = HJ;
    int init_f32 = bf16 ? 0 : 1;
    if (mode == Mode::FROM_CARRIES) {
        init_p = carries;
        init_stride = ((S + QS_CARRY_STEPS - 1) / QS_CARRY_STEPS) * HJ;
        init_f32 = 1;
    }
    qs::Geometry geo = pl.geo;
    float4 *save4 = mode == Mode::SAVE_CARRIES ? reinterpret_cast<float4 *>(carries) : nullptr;
    const void *q4 = q, *d4 = d_cum;
    void *out4 = out, *dinit4 = d_init;
    void *fwd_args[] = {&q4, &init_p, &init_stride, &init_f32, &out4, &save4, &geo};
    void *bwd_args[] = {&q4, &d4, &init_p, &init_stride, &init_f32, &out4, &dinit4, &geo};
    if (cudaLaunchKernel(pl.v->agg, dim3((unsigned)geo.NG), dim3(pl.v->threads()), bwd ? bwd_args : fwd_args, 0,
                         stream) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
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
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    Plan pl;
    rc = make_plan(bwd, B, S, HJ, di->sms, &pl, mode, bf16, cs != cudaStreamCaptureStatusNone);
    if (rc != QS_OK) return rc;
    unsigned char *ws = nullptr;
    rc = ensure_workspace(dev, stream, pl.ws_bytes, &ws);
    if (rc != QS_OK) return rc;
    if (pl.v->smax > 0)
        return launch_short(pl, bwd, q, d_cum, out, init, d_init, S, HJ, stream, mode, carries, bf16);
    CUtensorMap qmap, dmap;
    const int eb = bf16 ? 8 : 16;
    rc = make_map(&qmap, q, B, S, HJ, pl.v->lt, pl.v->T(), eb);
    if (rc == QS_OK) rc = make_map(&dmap, bwd ? d_cum : q, B, S, HJ, pl.v->lt, pl.v->T(), eb);
    if (rc != QS_OK) return rc;
    if (pl.v->segk > 0 && bwd) return launch_segwalk_bwd(pl, dev, ws, q, d_cum, out, init, d_init, B, S, HJ, stream,
                                                           mode, carries, bf16);
    if (pl.v->segk > 0) {
        uint32_t epoch = 0, *flags = nullptr;
        rc = chain_flags(dev, stream, pl.o_L, &flags, &epoch);
        if (rc != QS_OK) return rc;
        int grid = 0;
        rc = persistent_grid(dev, pl.v, &grid);
        if (rc != QS_OK) return rc;
        const long long units = (long long)pl.geo.NG * ((pl.geo.C + pl.v->segk - 1) / pl.v->segk);
        if (grid > units) grid = (int)units;
        qs::Control ctl = control_block(ws, true);
        const void *init4 = init;
        void *out4 = out;
        float4 *save4 = mode == Mode::SAVE_CARRIES ? reinterpret_cast<float4 *>(carries) : nullptr;
        unsigned int *tickets = flags;   // counters, zero between launches
        uint32_t *status = flags + kFlagsHead / 4;
        float4 *aggv = reinterpret_cast<float4 *>(ws + pl.o_W);
        float4 *inclv = reinterpret_cast<float4 *>(ws + pl.o_F);
        float4 *agg_next = nullptr, *incl_next = nullptr;
        std::unique_lock<std::mutex> order(g_lbv_launch_mu, std::defer_lock);
        if (pl.v->sent) {
            order.lock();
            float4 *cur[kLbMaxArrays], *nxt[kLbMaxArrays];
            rc = lb_values(dev, stream, LB_FWD, units * pl.v->lt, 2, cur, nxt);
            if (rc != QS_OK) return rc;
            aggv = cur[0];
            inclv = cur[1];
            agg_next = nxt[0];
            incl_next = nxt[1];
        }
        void *args[] = {&qmap, &init4, &out4, &save4, &status, &tickets, &aggv, &inclv, &agg_next, &incl_next,
                        &pl.geo, &ctl, &epoch};
        void *tab_args[] = {&qmap, &init4, &out4, &save4, &tickets, &aggv, &inclv, &agg_next, &incl_next, &pl.geo, &ctl};
        if (cudaLaunchKernel(pl.v->agg, dim3((unsigned)grid), dim3(pl.v->threads()), pl.v->tab ? tab_args : args,
                             pl.v->smem(), stream) != cudaSuccess) {
            cudaGetLastError();
            if (pl.v->sent) lb_values_invalidate(dev, stream, LB_FWD);
            return QS_ERR_CUDA;
        }
        return QS_OK;
    }
    if (pl.v->chain) {
        uint32_t epoch = 0, *flags = nullptr;
        rc = chain_flags(dev, stream, pl.o_L, &flags, &epoch);
        if (rc != QS_OK) return rc;
        flags += kFlagsHead / 4;   // past the ticket counter
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
        void **args = bwd ? bwd_args : fwd_args;
        if (cudaLaunchKernel(pl.v->agg, dim3((unsigned)pl.walk_grid), dim3(pl.v->threads()), args, pl.v->smem(),
                             stream) != cudaSuccess) {
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
    // Many chunks per lane: kCarryScanLanes lanes per block and a scan over
    // 256 / kCarryScanLanes chunk ranges per lane.
    constexpr int LPB = kCarryScanLanes;
    const bool scan = pl.geo.C > 256;
    if (scan) {
        carry_fn = bf16 ? (bwd ? reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoBF16, true, LPB>)
                               : reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoBF16, false, LPB>))
                        : (bwd ? reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoF32, true, LPB>)
                               : reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoF32, false, LPB>));
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
    const int carry_blocks = scan ? (pl.geo.NL + LPB - 1) / LPB : (pl.geo.NL + pl.carry_lb - 1) / pl.carry_lb;
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

// ===========================================================================
// quat_cumprod_fwd_bwd_host: one forward + backward step on host buffers.
// The work is cut into slices (whole batch entries, or lane ranges of one
// entry when an entry is large; lanes are independent); slice i is copied in
// on an internal stream while slice i-1 is computed on the caller's stream
// and slice i-2 is copied out on a second internal stream, through NSLOT
// device staging slots (a slot is reused once its copy-out is done).  The
// caller's stream waits for the last copy-out, so the call is ordered like
// cudaMemcpyAsync: prior work on `stream` first, and the host outputs are
// ready once `stream` has been synchronized.
// ===========================================================================
namespace {

constexpr int NSLOT = 3;
constexpr size_t kSliceBytes = 32u << 20;   // about this much of one tensor per slice

struct HostPipe {
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_done[NSLOT] = {}, comp_done[NSLOT] = {}, out_done[NSLOT] = {};
    unsigned char *stage = nullptr;
    size_t bytes = 0;
};
std::map<int, HostPipe> g_pipe;
std::mutex g_pipe_mu;   // one host-buffer step enqueued at a time per process

int pipe_of(int dev, size_t slot_bytes, HostPipe **out) {
    HostPipe &p = g_pipe[dev];
    if (!p.ready) {
        bool ok = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&p.end, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < NSLOT; ++i)
            ok = cudaEventCreateWithFlags(&p.in_done[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.comp_done[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.out_done[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        p.ready = true;
    }
    const size_t need = slot_bytes * NSLOT;
    if (p.bytes < need) {
        // Earlier steps may still copy out of the old staging: wait for them.
        if (cudaStreamSynchronize(p.s_in) != cudaSuccess || cudaStreamSynchronize(p.s_out) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        if (p.stage) cudaFree(p.stage);
        p.stage = nullptr;
        p.bytes = 0;
        void *m = nullptr;
        if (cudaMalloc(&m, need) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_NOMEM;
        }
        p.stage = static_cast<unsigned char *>(m);
        p.bytes = need;
    }
    *out = &p;
    return QS_OK;
}

}  // namespace

extern "C" int quat_cumprod_fwd_bwd_host(const float *q, const float *init, const float *d_cum, float *cum,
                                         float *d_q, float *d_init, int64_t B, int64_t S, int64_t H, int64_t J,
                                         void *stream_) {
    const int dc = check_dims(B, S, H, J);
    if (dc != QS_OK && dc != 1) return dc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const int64_t HJ = H * J;
    if (dc == 1) {
        // No steps but some lanes: the gradient of init is zero (written once
        // the work already on the stream is done).
        if (S == 0 && B > 0 && HJ > 0) {
            if (!d_init) return QS_ERR_NULL;
            if (cudaStreamSynchronize(stream) != cudaSuccess) {
                cudaGetLastError();
                return QS_ERR_CUDA;
            }
            std::memset(d_init, 0, (size_t)B * HJ * 16);
        }
        return QS_OK;
    }
    if (!q || !init || !d_cum || !cum || !d_q || !d_init) return QS_ERR_NULL;
    const size_t big = (size_t)B * S * HJ * 16, small = (size_t)B * HJ * 16;
    const void *ins[3] = {q, init, d_cum};
    const size_t insz[3] = {big, small, big};
    const void *outs[3] = {cum, d_q, d_init};
    const size_t outsz[3] = {big, big, small};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 3; ++i)
            if (overlaps(outs[o], outsz[o], ins[i], insz[i])) return QS_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlaps(outs[o], outsz[o], outs[o2], outsz[o2])) return QS_ERR_ALIAS;
    }
    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;

    // Slices: whole batch entries, about kSliceBytes of a tensor each.  With
    // fewer than kMinEntries entries there would be too little to overlap:
    // then lane ranges of one entry (pitched copies) of at least kMinLanes
    // lanes, up to kRanges ranges per entry.  Rows of 512 bytes (32 lanes)
    // copy at the link's rate; 256-byte rows made the 1 x 131072 x 16 x 16
    // step 37% slower, 1 KiB rows (fewer, larger ranges) 2% slower.
    constexpr int64_t kMinEntries = 4, kMinLanes = 32, kRanges = 8;
    const size_t per_b = (size_t)S * HJ * 16;
    const bool by_lanes = B < kMinEntries && HJ >= 2 * kMinLanes;
    const int64_t sb = by_lanes ? 1 : std::max<int64_t>(1, std::min<int64_t>(B, (int64_t)(kSliceBytes / per_b)));
    int64_t sl_even = HJ;
    if (by_lanes) {
        const int64_t ranges = std::min<int64_t>(kRanges / B < 2 ? 2 : kRanges / B, HJ / kMinLanes);
        sl_even = (HJ + ranges - 1) / ranges;
        sl_even = (sl_even + 15) / 16 * 16;   // 256-byte rows
    }
    // One staging slot: q, d_cum, cum, d_q of a slice, then init and d_init.
    const size_t big_s = align_up((size_t)sb * S * sl_even * 16, 256), small_s = align_up((size_t)sb * sl_even * 16, 256);
    const size_t slot_bytes = 4 * big_s + 2 * small_s;

    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe *p = nullptr;
    rc = pipe_of(dev, slot_bytes, &p);
    if (rc != QS_OK) return rc;
    auto fail = [&]() {
        cudaGetLastError();
        return QS_ERR_CUDA;
    };
    // Nothing starts before the work already on the caller's stream.
    if (cudaEventRecord(p->start, stream) != cudaSuccess || cudaStreamWaitEvent(p->s_in, p->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(p->s_out, p->start, 0) != cudaSuccess)
        return fail();
    const unsigned char *hq = reinterpret_cast<const unsigned char *>(q);
    const unsigned char *hi = reinterpret_cast<const unsigned char *>(init);
    const unsigned char *hd = reinterpret_cast<const unsigned char *>(d_cum);
    unsigned char *hc = reinterpret_cast<unsigned char *>(cum);
    unsigned char *hg = reinterpret_cast<unsigned char *>(d_q);
    unsigned char *hgi = reinterpret_cast<unsigned char *>(d_init);
    const size_t row = (size_t)HJ * 16;   // one step of one batch entry in the host tensors
    int i = 0;
    for (int64_t b0 = 0; b0 < B; b0 += sb) {
        const int64_t nb = std::min<int64_t>(sb, B - b0);
        for (int64_t l0 = 0; l0 < HJ; l0 += sl_even, ++i) {
            const int64_t nl = std::min<int64_t>(sl_even, HJ - l0);
            const int slot = i % NSLOT;
            unsigned char *base = p->stage + (size_t)slot * slot_bytes;
            float *sq = reinterpret_cast<float *>(base), *sd = reinterpret_cast<float *>(base + big_s);
            float *sc = reinterpret_cast<float *>(base + 2 * big_s), *sg = reinterpret_cast<float *>(base + 3 * big_s);
            float *si = reinterpret_cast<float *>(base + 4 * big_s);
            float *sgi = reinterpret_cast<float *>(base + 4 * big_s + small_s);
            const size_t w = (size_t)nl * 16;                  // bytes of one step of the slice
            const size_t hoff = (size_t)b0 * S * row + (size_t)l0 * 16;
            const size_t ioff = (size_t)b0 * row + (size_t)l0 * 16;
            const size_t rows = (size_t)nb * S;                // whole entries: rows of `row` bytes
            // in: once the slot's previous copy-out is done
            auto in2d = [&](void *dst, const unsigned char *src, size_t height) {
                return cudaMemcpy2DAsync(dst, w, src, row, w, height, cudaMemcpyHostToDevice, p->s_in) == cudaSuccess;
            };
            auto out2d = [&](unsigned char *dst, const void *src, size_t height) {
                return cudaMemcpy2DAsync(dst, row, src, w, w, height, cudaMemcpyDeviceToHost, p->s_out) == cudaSuccess;
            };
            if (cudaStreamWaitEvent(p->s_in, p->out_done[slot], 0) != cudaSuccess || !in2d(sq, hq + hoff, rows) ||
                !in2d(si, hi + ioff, (size_t)nb) || !in2d(sd, hd + hoff, rows) ||
                cudaEventRecord(p->in_done[slot], p->s_in) != cudaSuccess)
                return fail();
            // compute on the caller's stream: nb entries of nl lanes
            if (cudaStreamWaitEvent(stream, p->in_done[slot], 0) != cudaSuccess) return fail();
            rc = launch(false, sq, nullptr, sc, si, nullptr, nb, S, nl, stream);
            if (rc == QS_OK) rc = launch(true, sq, sd, sg, si, sgi, nb, S, nl, stream);
            if (rc != QS_OK) return rc;
            if (cudaEventRecord(p->comp_done[slot], stream) != cudaSuccess) return fail();
            // out
            if (cudaStreamWaitEvent(p->s_out, p->comp_done[slot], 0) != cudaSuccess || !out2d(hc + hoff, sc, rows) ||
                !out2d(hg + hoff, sg, rows) || !out2d(hgi + ioff, sgi, (size_t)nb) ||
                cudaEventRecord(p->out_done[slot], p->s_out) != cudaSuccess)
                return fail();
        }
    }
    // The caller's stream waits for the last copy-out (s_out runs in order).
    if (cudaEventRecord(p->end, p->s_out) != cudaSuccess || cudaStreamWaitEvent(stream, p->end, 0) != cudaSuccess)
        return fail();
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
    // The stream's workspace, and the device's no-alloc scratch (set up by a
    // quat_cumprod_bwd_noalloc call on this device); neither is allocated here.
    unsigned char *bases[2] = {nullptr, nullptr};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_ws.find({dev, reinterpret_cast<uintptr_t>(stream)});
        if (it != g_ws.end()) bases[0] = it->second.base;
        auto na = g_noalloc_ptr.find(dev);
        if (na != g_noalloc_ptr.end()) bases[1] = na->second;
    }
    int status = QS_OK;
    for (unsigned char *base : bases) {
        if (!base) continue;
        qs::WsHeader h;
        if (cudaMemcpy(&h, base, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        if (h.err_code == 0) continue;
        if (cudaMemset(base, 0, sizeof(qs::WsHeader)) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        status = QS_ERR_TIMEOUT;
    }
    return status;
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
    if (pl.v->segk > 0 && bwd) *kernels = mode == Mode::FROM_CARRIES ? 1 : 2;   // (+ the carries-only pass)
    else *kernels = (pl.v->walk || pl.v->chain || pl.v->segk > 0 || pl.v->smax > 0) ? 1 : (mode == Mode::SAVE_CARRIES ? 4 : 3);
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

extern "C" int quat_cumprod_debug_set_walk_cap(int64_t ctas) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_bwd_cap = (ctas <= 0 || ctas > INT32_MAX) ? -1 : (int)ctas;
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

// Address of the scratch on the current device `dev`, looked up once per
// device (the lookup loads this library's device code on that device).  The
// lookup is refused while `stream` is being captured (QS_ERR_NOMEM, as for a
// workspace that would have to be set up during a capture).
int noalloc_scratch(int dev, cudaStream_t stream, unsigned char **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_noalloc_ptr.find(dev);
    if (it != g_noalloc_ptr.end()) {
        *out = it->second;
        return QS_OK;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return QS_ERR_NOMEM;
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
    // The first call on a device sets up the library there (kernel
    // attributes, the array's address): not while the stream is captured.
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return QS_ERR_CUDA;
    }
    bool ready;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ready = g_noalloc_ptr.count(cur) != 0;
    }
    if (!ready) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
            cudaGetLastError();
            return QS_ERR_CUDA;
        }
        if (cs != cudaStreamCaptureStatusNone) return QS_ERR_NOMEM;
    }
    DevInfo *di = nullptr;
    int dev = 0;
    int rc = device_info(&di, &dev);
    if (rc != QS_OK) return rc;
    unsigned char *ws = nullptr;
    rc = noalloc_scratch(dev, stream, &ws);
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

    // Every aggregate and carry slot a call reads is written earlier in the
    // same call.  The status block starts at zero (the array is zeroed when
    // the library's device code is loaded) and keeps a timeout until
    // quat_cumprod_status reads and clears it, as a stream's workspace does.
    CUtensorMap qmap, dmap;
    rc = make_map(&qmap, q, B, S, HJ, NA_LT, NA_T);
    if (rc == QS_OK) rc = make_map(&dmap, d_cum, B, S, HJ, NA_LT, NA_T);
    if (rc != QS_OK) return rc;
    qs::Control ctl = control_block(ws, true);
    const float4 *init4 = reinterpret_cast<const float4 *>(init);
    float4 *dinit4 = reinterpret_cast<float4 *>(d_init);
    float4 *out4 = reinterpret_cast<float4 *>(d_q);
    const float4 *aggL_c = aggL, *aggW_c = aggW, *carF_c = carF, *carH_c = carH;
    int lt = NA_LT;
    // The carry step as in quat_cumprod_bwd: 32 lanes per block up to 256
    // chunks per lane, beyond that the scan over chunk ranges, kCarryScanLanes
    // lanes per block.
    const bool scan = geo.C > 256;
    const int carry_lb = scan ? kCarryScanLanes : 32;
    const void *agg_fn = reinterpret_cast<const void *>(qs::quat_agg_kernel<qs::IoF32, true, NA_LT, NA_N>);
    const void *apply_fn = reinterpret_cast<const void *>(qs::quat_apply_kernel<qs::IoF32, true, NA_LT, NA_N>);
    const void *carry_fn =
        scan ? reinterpret_cast<const void *>(qs::quat_carry_scan_kernel<qs::IoF32, true, kCarryScanLanes>)
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
