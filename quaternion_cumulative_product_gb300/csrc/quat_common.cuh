// quat_common.cuh -- what every kernel of the scan shares: the workspace status block,
// the geometry of a call, the control block of the bounded waits, and the
// staging of one tile by TMA.
#pragma once

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

}  // namespace qs
