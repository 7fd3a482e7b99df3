// quat_device.cuh -- device-side building blocks of the quaternion scan:
// Hamilton-product arithmetic on float4 and the sm_100-family PTX used by the
// kernels (mbarrier, TMA tensor loads and stores, bulk async-groups,
// acquire/release flags, global timer).
//
// Quaternion layout: float4 (x, y, z, w) holds [w, x, y, z] of the quaternion,
// i.e. .x is the real part and .y/.z/.w are the i/j/k parts, matching the
// [..., 4] = [w, x, y, z] memory layout of the tensors.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace qs {

// ---------------------------------------------------------------------------
// Quaternion arithmetic (Hamilton convention, i^2 = j^2 = k^2 = ijk = -1).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 q_ident() { return make_float4(1.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ float4 q_zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ float4 q_nan() {
    const float n = __int_as_float(0x7fc00000);
    return make_float4(n, n, n, n);
}

__device__ __forceinline__ float4 q_conj(const float4 a) { return make_float4(a.x, -a.y, -a.z, -a.w); }

__device__ __forceinline__ float4 q_add(const float4 a, const float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// a (x) b
__device__ __forceinline__ float4 q_mul(const float4 a, const float4 b) {
    float4 r;
    r.x = a.x * b.x - a.y * b.y - a.z * b.z - a.w * b.w;
    r.y = a.x * b.y + a.y * b.x + a.z * b.w - a.w * b.z;
    r.z = a.x * b.z - a.y * b.w + a.z * b.x + a.w * b.y;
    r.w = a.x * b.w + a.y * b.z - a.z * b.y + a.w * b.x;
    return r;
}

// conj(a) (x) b  and  a (x) conj(b); the negations fold into the FMAs.
__device__ __forceinline__ float4 q_mul_cl(const float4 a, const float4 b) { return q_mul(q_conj(a), b); }
__device__ __forceinline__ float4 q_mul_cr(const float4 a, const float4 b) { return q_mul(a, q_conj(b)); }

// acc + a (x) b and acc + conj(a) (x) b, accumulated term by term into acc
// (four fused multiply-adds per component).
__device__ __forceinline__ float4 q_fma(const float4 acc, const float4 a, const float4 b) {
    float4 r;
    r.x = fmaf(-a.w, b.w, fmaf(-a.z, b.z, fmaf(-a.y, b.y, fmaf(a.x, b.x, acc.x))));
    r.y = fmaf(-a.w, b.z, fmaf(a.z, b.w, fmaf(a.y, b.x, fmaf(a.x, b.y, acc.y))));
    r.z = fmaf(a.w, b.y, fmaf(a.z, b.x, fmaf(-a.y, b.w, fmaf(a.x, b.z, acc.z))));
    r.w = fmaf(a.w, b.x, fmaf(-a.z, b.y, fmaf(a.y, b.z, fmaf(a.x, b.w, acc.w))));
    return r;
}
__device__ __forceinline__ float4 q_fma_cl(const float4 acc, const float4 a, const float4 b) {
    return q_fma(acc, q_conj(a), b);
}

// ---------------------------------------------------------------------------
// Element types of the tensors in memory.  Arithmetic is always fp32; an I/O
// type says how one quaternion is stored and converts it.
// ---------------------------------------------------------------------------
struct IoF32 {             // four fp32, 16 bytes
    using elem = float4;
    static constexpr uint32_t bytes = 16;
    __device__ __forceinline__ static float4 get(const elem &v) { return v; }
    __device__ __forceinline__ static elem put(const float4 v) { return v; }
};

struct IoBF16 {            // four bfloat16 [w, x, y, z], 8 bytes
    using elem = uint2;
    static constexpr uint32_t bytes = 8;
    __device__ __forceinline__ static float4 get(const elem &v) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    __device__ __forceinline__ static elem put(const float4 v) {   // round to nearest even
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        elem r;
        r.x = *reinterpret_cast<const uint32_t *>(&a);
        r.y = *reinterpret_cast<const uint32_t *>(&b);
        return r;
    }
};

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and TMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Block barrier among the first `nthreads` threads (named barrier `id`).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so
// that they all take the same branch afterwards.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// 3-D tiled TMA load of the box at (x, y, z) into shared memory; completion is
// signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// 4-D tiled TMA load of the box at (x, y, z, w).
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
        : "memory");
}

// 4-D tiled TMA store of a shared-memory box to (x, y, z, w).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int x, int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(src))
        : "memory");
}

// 3-D tiled TMA store of a shared-memory box to (x, y, z); out-of-range parts
// of the box are not written.  Completion is tracked by bulk async-groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_addr(src))
        : "memory");
}

// Same load with an L2 cache policy (from createpolicy) for the copied lines.
__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map, int x, int y, int z,
                                                 uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policies: keep the lines (they are read again soon) or drop them first.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N of this thread's bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Asynchronous 16-byte copy global -> shared (cp.async, L2 only); completion
// by cp_async_wait_all in the issuing thread.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// GPU-scope flags and the global timer.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Turns earlier relaxed loads that observed release stores into acquires.
__device__ __forceinline__ void fence_acquire_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const unsigned int *p) {
    return *reinterpret_cast<const volatile unsigned int *>(p);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace qs
