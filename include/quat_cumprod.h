/*
 * quat_cumprod.h -- C ABI of the GB300 (sm_103a) quaternion cumulative-product
 * scan and its recompute-based backward.
 *
 * The operation is the one defined in burn-mamba `mamba3/quat_scan/backward.rs`,
 * module documentation, section "Gradient math":
 *
 *     cum[t] = q_t (x) cum[t-1],     cum[-1] = init            (forward)
 *
 * and, for a cotangent d_cum of cum, the vector-Jacobian product
 *
 *     G[t]   = d_cum[t] + conj(q_{t+1}) (x) G[t+1]               (reverse recurrence)
 *     d_q[t] = G[t] (x) conj(cum[t-1])
 *     d_init = conj(q_0) (x) G[0]   (= the page's S[0] for every non-zero q_0)
 *
 * which for unit quaternions is the page's closed form with the prefix product
 * P_t = q_t (x) ... (x) q_0 and the suffix sum S[t] = sum_{s>=t} conj(P_s) (x) d_cum[s].
 * (x) is the Hamilton product (i^2 = j^2 = k^2 = ijk = -1); a quaternion is four
 * floats [w, x, y, z].  As on the page, the backward takes only the leaves
 * (q, init) and the cotangent: nothing is saved between forward and backward.
 * The backward is exact for all quaternions, not only unit ones.
 *
 * Layout (all tensors): contiguous row-major fp32.
 *   q, cum, d_cum, d_q : [B, S, H, J, 4]   element (b,s,h,j) at float offset
 *                                          (((b*S + s)*H + h)*J + j)*4
 *   init, d_init       : [B, H, J, 4]
 * A "lane" is one (b, h, j); lanes are independent, the scan runs along s.
 *
 * Pointers: device pointers (cudaMalloc / torch CUDA memory) on the current
 * device, owned by the caller, never freed or retained by the library, each
 * aligned to 16 bytes.  Outputs must not overlap inputs.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 * Every call is asynchronous: it validates arguments, enqueues its work on
 * `stream` and returns.  Launch failures are returned at once; a failure that
 * happens on the device (a wait that ran out) is recorded in a per-stream
 * device word and reported by quat_cumprod_status().
 *
 * Scratch memory: the calls use a library-owned workspace per (device,
 * stream) for a status block and per-chunk aggregates and carries.  Per lane
 * and 64-step chunk this is nothing for a forward walk or the short-sequence
 * kernels (at most 2048 steps, the whole sequence of a few lanes in one CTA),
 * 16 bytes for a backward walk or the backward's segmented walk, and 32
 * (forward) or 64 (backward) bytes for the aggregate / carry / apply kernels
 * (see quat_cumprod_plan for which a call uses).  The segmented chained walks
 * (for few lane groups) keep, per lane and segment of 2 to 8 chunks, two copies
 * of 32 (forward) or 48 (backward) bytes of look-back values plus a few
 * counters in further per-stream allocations, and reserve the aggregate /
 * carry / apply workspace of the same direction as well.  The first call on a
 * stream, and any later call that needs more scratch, allocates it
 * (cudaMalloc) and synchronizes that stream; issue such a call before
 * capturing the stream into a CUDA graph.  While a stream is being captured
 * the segmented walks give way to the aggregate / carry / apply kernels,
 * which keep no state from one launch to the next (the segmented walks'
 * look-back values are tied to the launch that reads them), so a captured
 * graph may be replayed any number of times; the walks and the
 * short-sequence kernels keep no state either.  Calls on one stream are ordered by the stream; calls on different
 * streams use different workspaces and may run concurrently.  A workspace is
 * found by the stream's handle: before destroying a stream, let its work
 * finish, so that a new stream given the same handle cannot meet a launch
 * still running on the old one's workspace.
 *
 * Sizes: B, S, H, J >= 0.  Any zero size makes the call a no-op that returns
 * QS_OK (except that quat_cumprod_bwd with S == 0 writes d_init = 0).
 * Limits: each of B, S, H, J below 2^31, S*H*J*16 < 2^40 bytes per batch
 * entry, H*J*4 < 2^32, the number of work tiles below 2^31.  A size past a
 * limit returns QS_ERR_DIMS before anything is enqueued.
 */
#ifndef QUAT_CUMPROD_H
#define QUAT_CUMPROD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum {
    QS_OK = 0,
    QS_ERR_NULL = -1,        /* a required pointer is NULL                      */
    QS_ERR_DIMS = -2,        /* a size is negative or beyond the limits above   */
    QS_ERR_MISALIGNED = -3,  /* a pointer is not 16-byte aligned                */
    QS_ERR_ALIAS = -4,       /* an output overlaps an input                     */
    QS_ERR_CUDA = -5,        /* a CUDA runtime call failed (launch, memset...)  */
    QS_ERR_TIMEOUT = -6,     /* a wait on the device ran out                    */
    QS_ERR_NOMEM = -7,       /* workspace allocation failed, or it would have to
                                grow while the stream is being captured         */
    QS_ERR_DEVICE = -8,      /* the current device is not compute capability 10.3 */
    QS_ERR_SCRATCH = -9      /* quat_cumprod_bwd_noalloc: the sizes need more
                                scratch than its fixed array holds              */
};

/*
 * Forward scan.  Reads q [B,S,H,J,4] and init [B,H,J,4]; writes
 * cum [B,S,H,J,4] with cum[b,s,h,j] = q[b,s,h,j] (x) cum[b,s-1,h,j] and
 * cum[b,-1,h,j] = init[b,h,j].
 * Definition: burn-mamba `mamba3/quat_scan/backward.rs`, "Gradient math"
 * (the scan), and `Mamba3QuatScanBackendExt::quat_cumprod(q_bshj4, init_bhj4)`.
 */
int quat_cumprod_fwd(const float *q, const float *init, float *cum,
                     int64_t B, int64_t S, int64_t H, int64_t J, void *stream);

/*
 * Backward (vector-Jacobian product) of the forward scan, recomputed from the
 * leaves.  Reads q, init and d_cum (the cotangent of cum, same shape as q);
 * writes d_q [B,S,H,J,4] and d_init [B,H,J,4] as defined at the top of this
 * file.  A cotangent of a "final carry" cum[:, S-1] must already be added
 * into d_cum[:, S-1] by the caller, as the page's module documentation says.
 * Definition: burn-mamba `mamba3/quat_scan/backward.rs`, "Gradient math"
 * (VJP rule, reverse recurrence, closed form) and `quat_scan_backward`.
 */
int quat_cumprod_bwd(const float *q, const float *init, const float *d_cum,
                     float *d_q, float *d_init,
                     int64_t B, int64_t S, int64_t H, int64_t J, void *stream);

/*
 * Backward without allocation: computes exactly what quat_cumprod_bwd
 * computes, with the same arguments, layout, ownership and checks, but never
 * allocates device memory.  The page has no counterpart: this entry point
 * exists for callers that cannot call cudaMalloc at the point where they need
 * the gradient, for example
 *   - code whose device memory is all handed out by another allocator (a
 *     framework's caching allocator, or a runtime with a fixed memory budget
 *     reserved at start-up), where a raw cudaMalloc can fail or fragment that
 *     allocator's pool;
 *   - latency-critical loops that cannot afford the device-wide
 *     synchronization that cudaFree implies (quat_cumprod_bwd may free and
 *     re-allocate its workspace when a call needs a larger one).
 * It calls no cudaMalloc, no cudaFree and no other allocating routine.
 *
 * Scratch: one fixed array of this library in device memory (a file-scope
 * __device__ variable), 16 MiB + 256 bytes on every device where the
 * library's kernels are loaded.  It holds a status block and the per-chunk
 * aggregates and carries of one call, so the sizes are limited to
 *     B * ceil(H*J / 32) * ceil(S / 64) <= QS_NOALLOC_MAX_TILES (8192)
 * work tiles (for example B=8, S=4096, H=16, J=32 fits exactly); larger sizes
 * return QS_ERR_SCRATCH before anything is enqueued.
 *
 * Every call on a device shares that one array.  Everything a call reads
 * from it (chunk aggregates and carries) it has written earlier in the same
 * call.  Calls whose work can overlap on the GPU (calls on different streams
 * without an ordering between them, or from several host threads onto
 * unordered streams) RACE on the array and give wrong results; calls on one
 * stream are ordered and safe.
 *
 * Set-up: the first call on each device looks up the array's address on that
 * device (cudaGetSymbolAddress, with that device current) and prepares the
 * kernels' attributes; later calls reuse both.  Make that first call on each
 * device before any stream capture begins: a first call on a stream that is
 * being captured returns QS_ERR_NOMEM and enqueues nothing.
 *
 * Errors as for quat_cumprod_bwd, plus QS_ERR_SCRATCH.  A device-side wait
 * that runs out (possible only if a tile's copy never lands) is recorded in
 * the array's own status block, which starts at zero when the library is
 * loaded on the device and keeps the record across calls:
 * quat_cumprod_status(stream) reads and clears it (besides the stream's own
 * record), allocating nothing, so call it with the stream the no-alloc calls
 * were enqueued on.  The debug stall hook applies as to quat_cumprod_bwd.
 */
#define QS_NOALLOC_MAX_TILES 8192
int quat_cumprod_bwd_noalloc(const float *q, const float *init, const float *d_cum,
                             float *d_q, float *d_init,
                             int64_t B, int64_t S, int64_t H, int64_t J, void *stream);

/*
 * Chunk carries.  A training step that keeps something between forward and
 * backward can skip the backward's recomputation of the forward carries: the
 * forward below also writes the state entering every QS_CARRY_STEPS-step
 * chunk,
 *
 *     carries[b, c, h, j] = cum[b, c*QS_CARRY_STEPS - 1, h, j]   (init for c = 0),
 *
 * an extra [B, ceil(S / QS_CARRY_STEPS), H, J, 4] fp32 tensor (1/64 of q),
 * and the backward below takes it in place of init.  The page's autodiff node
 * deliberately keeps only q and init (burn-mamba `mamba3/quat_scan/backward.rs`,
 * `QuatScanBackward` / `State`: the leaves, no scan intermediates); these two
 * calls are the variant that keeps the carries as well, so that the backward
 * reads q once instead of twice.  Results equal quat_cumprod_fwd and
 * quat_cumprod_bwd (with init = carries[:, 0]) up to rounding order.
 */
#define QS_CARRY_STEPS 64

/*
 * Forward scan that also writes `carries` (device, caller-owned, 16-byte
 * aligned, overlapping nothing else).  Arguments, layout and errors otherwise
 * as quat_cumprod_fwd.
 */
int quat_cumprod_fwd_carries(const float *q, const float *init, float *cum, float *carries,
                             int64_t B, int64_t S, int64_t H, int64_t J, void *stream);

/*
 * Backward from the carries written by quat_cumprod_fwd_carries for the same
 * q and init: writes d_q and d_init as quat_cumprod_bwd(q, carries[:, 0],
 * d_cum) would, reading q and d_cum once (the walk, or for too few lane
 * groups the segmented walk, takes every chunk's carry from `carries`; the
 * short-sequence kernels, which hold the whole sequence anyway, and the
 * aggregate / carry / apply kernels, which a debug setting can force, use
 * them only as init).  Arguments, layout and errors otherwise as
 * quat_cumprod_bwd.
 */
int quat_cumprod_bwd_carries(const float *q, const float *carries, const float *d_cum,
                             float *d_q, float *d_init,
                             int64_t B, int64_t S, int64_t H, int64_t J, void *stream);

/*
 * bfloat16 I/O.  The same scan and backward with every tensor (q, init, cum,
 * d_cum, d_q, d_init) in bfloat16: a quaternion is four bfloat16 bit patterns
 * [w, x, y, z] (8 bytes, passed as uint16_t), laid out as above.  The
 * arithmetic is fp32 throughout (chunk carries included); each output is
 * rounded to the nearest bfloat16 (ties to even) once, when it is stored, so
 * an output differs from the exact result for the bfloat16 inputs by at most
 * half a bfloat16 ulp (2^-8 of its magnitude) plus the fp32 error of the fp32
 * calls.  Requires
 * H*J even (TMA row strides are multiples of 16 bytes; QS_ERR_DIMS
 * otherwise); pointers 16-byte aligned.  The designs follow the fp32 calls'
 * choice by size (quat_cumprod_plan, calls 4 and 5).
 * The pages define the scan in full precision; this halves the bytes moved
 * (8 bytes per quaternion instead of 16).
 */
int quat_cumprod_fwd_bf16(const uint16_t *q, const uint16_t *init, uint16_t *cum,
                          int64_t B, int64_t S, int64_t H, int64_t J, void *stream);
int quat_cumprod_bwd_bf16(const uint16_t *q, const uint16_t *init, const uint16_t *d_cum,
                          uint16_t *d_q, uint16_t *d_init,
                          int64_t B, int64_t S, int64_t H, int64_t J, void *stream);

/*
 * One forward + backward step on HOST buffers: cum = the forward scan of
 * (q, init), and (d_q, d_init) = its backward from d_cum, exactly what
 * quat_cumprod_fwd and quat_cumprod_bwd compute, with the same layouts, but
 * every pointer is host memory (page-locked memory lets the copies overlap;
 * other host memory works, with the copies serialised).  No alignment is
 * required.  The batch is processed in slices of whole batch entries:
 * the copy of slice i to the device, the kernels of slice i-1 (on `stream`)
 * and the copy of slice i-2 back overlap, through library-owned device
 * staging (grown as needed, kept for later calls).
 * Ordering is that of cudaMemcpyAsync: nothing starts before the work
 * already on `stream`, and the host outputs are complete once `stream` has
 * been synchronized (quat_cumprod_status(stream) does that and reports
 * device-side errors of the step).  The caller must not touch the host
 * buffers before then.
 * Errors as for quat_cumprod_bwd, except QS_ERR_MISALIGNED; QS_ERR_ALIAS if
 * an output overlaps an input or another output.
 */
int quat_cumprod_fwd_bwd_host(const float *q, const float *init, const float *d_cum,
                              float *cum, float *d_q, float *d_init,
                              int64_t B, int64_t S, int64_t H, int64_t J, void *stream);

/*
 * Synchronizes `stream`, then returns QS_ERR_TIMEOUT if any call enqueued on it
 * since the previous quat_cumprod_status() recorded a device-side timeout
 * (its outputs are then invalid), QS_ERR_CUDA if the synchronization failed,
 * and QS_OK otherwise.  Clears the recorded error.  It also reads and clears
 * the record of quat_cumprod_bwd_noalloc's scratch on the current device (one
 * record per device, shared by every stream).  It allocates nothing.
 */
int quat_cumprod_status(void *stream);

/*
 * Which compiled configuration a call with these sizes would use on the
 * current device, and how many kernels it launches: 1 for a walk (one CTA
 * per lane group streams the whole sequence), a segmented walk (too few
 * lane groups: the sequence cut into segments chained by look-back) or the
 * short-sequence kernels (at most 2048 steps: the whole sequence of a few
 * lanes in one CTA), 2 for the backward's segmented walk after its
 * carries-only pass, 3 for aggregate / carry / apply (independent tiles),
 * plus 1 when the forward exports its carries from that path.  `call`: 0 quat_cumprod_fwd, 1 quat_cumprod_bwd,
 * 2 quat_cumprod_fwd_carries, 3 quat_cumprod_bwd_carries, 4 quat_cumprod_fwd_bf16,
 * 5 quat_cumprod_bwd_bf16.  Writes
 * *variant = -1 and *kernels = 0 when the call would launch nothing.  Returns
 * the status the call's size and device checks would return (QS_ERR_DIMS for
 * an unknown `call`).  Nothing is enqueued.
 */
int quat_cumprod_plan(int call, int64_t B, int64_t S, int64_t H, int64_t J, int *variant, int *kernels);

/* Static, human-readable description of a status code. */
const char *quat_cumprod_strerror(int status);

/*
 * Test hooks.  quat_cumprod_debug_set_timeout_ns sets the limit of every
 * device-side wait (default 2 s; values <= 0 restore it).
 * quat_cumprod_debug_stall_tile(k) makes the first kernel of every later call
 * wait in tile k for bytes that never arrive (k < 0 disables), so that the
 * wait runs out its limit and the call reports QS_ERR_TIMEOUT instead of
 * hanging.  quat_cumprod_debug_set_variant selects a compiled tile
 * configuration for each direction (index into the library's variant table,
 * -1 = default; QS_ERR_DIMS for an unknown index).
 * quat_cumprod_debug_set_walk_cap(n) caps the CTAs of the backward walk
 * kernels at n (n <= 0 restores each configuration's own cap); the lane
 * groups are then walked in equal waves of at most n.  It caps the
 * persistent grid of the backward's segmented walk as well.  All four are
 * process-wide settings and return QS_OK unless stated.
 */
int quat_cumprod_debug_set_timeout_ns(int64_t ns);
int quat_cumprod_debug_stall_tile(int64_t tile);
int quat_cumprod_debug_set_variant(int fwd_variant, int bwd_variant);
int quat_cumprod_debug_set_walk_cap(int64_t ctas);
/* The same for the bfloat16 calls (their own table of configurations). */
int quat_cumprod_debug_set_variant_bf16(int fwd_variant, int bwd_variant);

#ifdef __cplusplus
}
#endif

#endif /* QUAT_CUMPROD_H */
