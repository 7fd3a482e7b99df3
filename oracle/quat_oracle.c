/*
 * quat_oracle.c -- fp64 CPU oracle for the quaternion cumulative-product scan.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the tests, the smoke
 * check of the entry module and the CPU-baseline leg of the benchmark load this
 * library.  It shares no code, header, table or helper with the CUDA library;
 * neither includes nor links the other.
 *
 * What it computes follows burn-mamba `mamba3/quat_scan/backward.rs`, module
 * documentation, section "Gradient math":
 *   - the scan         cum[t] = q_t (x) cum[t-1],   cum[-1] = init;
 *   - the per-factor VJP rule of o = a (x) b:  grad_a = g (x) conj(b),
 *                                              grad_b = conj(a) (x) g;
 *   - the reverse recurrence  G[t] = d_cum[t] + conj(q_{t+1}) (x) G[t+1];
 *   - the closed form for unit quaternions  S[t] = sum_{s>=t} conj(P_s) (x) d_cum[s],
 *     G[t] = P_t (x) S[t], d_q[t] = G[t] (x) conj(cum[t-1]), d_init = S[0].
 *
 * Readings where the page is silent (each is also listed in the design notes):
 *   - (x) is the Hamilton product (i^2 = j^2 = k^2 = ijk = -1), components are
 *     stored [w, x, y, z] (the page's `Quat` has a `.w` field);
 *   - the new factor multiplies on the LEFT (cum[t] = q_t (x) cum[t-1]);
 *   - cum holds cum[0..S-1] (init is not part of the output);
 *   - d_init of the literal recurrence is conj(q_0) (x) G[0], i.e. the VJP rule's
 *     grad_b applied to cum[0] = q_0 (x) init.  It equals the page's S[0] for
 *     every non-zero q_0: the cotangent of init is S[0] exactly, since
 *     cum[s] = P_s (x) init.
 *
 * Layout: q, cum, d_cum, d_q are contiguous row-major [B,S,H,J,4]; init and
 * d_init are [B,H,J,4].  A "lane" is one (b,h,j); lanes are independent, and the
 * only parallelism here is one POSIX thread per block of lanes.  Inside a lane
 * every loop runs sequentially over t in the page's order, in fp64, without
 * fast-math.  Inputs are fp64 (callers widen fp32 data before calling).
 *
 * Return value of every entry point: 0 on success, -1 on a bad argument
 * (negative size, NULL pointer with a non-zero size), -2 when a per-thread
 * buffer cannot be allocated.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------------------
 * Quaternion algebra, written out component by component.
 * ------------------------------------------------------------------------- */

/* out = a (x) b, Hamilton convention, [w,x,y,z]. */
static void hamilton(const double *a, const double *b, double *out)
{
    const double aw = a[0], ax = a[1], ay = a[2], az = a[3];
    const double bw = b[0], bx = b[1], by = b[2], bz = b[3];
    out[0] = aw * bw - ax * bx - ay * by - az * bz;
    out[1] = aw * bx + ax * bw + ay * bz - az * by;
    out[2] = aw * by - ax * bz + ay * bw + az * bx;
    out[3] = aw * bz + ax * by - ay * bx + az * bw;
}

/* out = conj(a) = (w, -x, -y, -z). */
static void conjugate(const double *a, double *out)
{
    out[0] = a[0];
    out[1] = -a[1];
    out[2] = -a[2];
    out[3] = -a[3];
}

void oracle_hamilton(const double *a, const double *b, double *out)
{
    double tmp[4];
    hamilton(a, b, tmp);
    memcpy(out, tmp, sizeof tmp);
}

void oracle_conj(const double *a, double *out)
{
    double tmp[4];
    conjugate(a, tmp);
    memcpy(out, tmp, sizeof tmp);
}

/* ---------------------------------------------------------------------------
 * Per-lane kernels.  `stride` is the distance, in quaternions, between t and
 * t+1 of one lane (H*J in the [B,S,H,J,4] layout).
 * ------------------------------------------------------------------------- */

/* Forward scan of one lane: c = init; for t: c = q[t] (x) c; cum[t] = c. */
static void lane_forward(const double *q, const double *init, double *cum,
                         int64_t S, int64_t stride)
{
    double c[4], next[4];
    memcpy(c, init, sizeof c);
    for (int64_t t = 0; t < S; ++t) {
        const double *qt = q + 4 * t * stride;
        hamilton(qt, c, next);
        memcpy(c, next, sizeof c);
        memcpy(cum + 4 * t * stride, c, sizeof c);
    }
}

/* Backward of one lane by the literal reverse recurrence.
 * cumbuf: scratch of 4*S doubles (this lane's cum, contiguous). */
static void lane_backward_recurrence(const double *q, const double *init,
                                     const double *d_cum, double *d_q,
                                     double *d_init, int64_t S, int64_t stride,
                                     double *cumbuf)
{
    if (S == 0) {
        memset(d_init, 0, 4 * sizeof(double));
        return;
    }
    /* Recompute cum[t] for t = 0..S-1. */
    double c[4], tmp[4];
    memcpy(c, init, sizeof c);
    for (int64_t t = 0; t < S; ++t) {
        hamilton(q + 4 * t * stride, c, tmp);
        memcpy(c, tmp, sizeof c);
        memcpy(cumbuf + 4 * t, c, sizeof c);
    }
    /* G[S-1] = d_cum[S-1]. */
    double G[4];
    memcpy(G, d_cum + 4 * (S - 1) * stride, sizeof G);
    for (int64_t t = S - 1; t >= 0; --t) {
        /* d_q[t] = G[t] (x) conj(cum[t-1]), cum[-1] = init
         * (VJP rule grad_a = g (x) conj(b) for cum[t] = q_t (x) cum[t-1]). */
        const double *prev = (t == 0) ? init : cumbuf + 4 * (t - 1);
        double cprev[4];
        conjugate(prev, cprev);
        hamilton(G, cprev, d_q + 4 * t * stride);
        /* Cotangent handed to cum[t-1] (VJP rule grad_b = conj(a) (x) g). */
        double cq[4], back[4];
        conjugate(q + 4 * t * stride, cq);
        hamilton(cq, G, back);
        if (t == 0) {
            memcpy(d_init, back, sizeof back);   /* d_init = conj(q_0) (x) G[0] */
        } else {
            /* G[t-1] = d_cum[t-1] + conj(q_t) (x) G[t]. */
            const double *d = d_cum + 4 * (t - 1) * stride;
            for (int k = 0; k < 4; ++k) G[k] = d[k] + back[k];
        }
    }
}

/* Backward of one lane by the page's closed form (exact for unit q only):
 *   P_t = q_t (x) P_{t-1} (P_{-1} = 1),  cum[t] = P_t (x) init,
 *   S[t] = sum_{s>=t} conj(P_s) (x) d_cum[s]   (reverse cumulative sum),
 *   G[t] = P_t (x) S[t],  d_q[t] = G[t] (x) conj(cum[t-1]),  d_init = S[0].
 * pbuf, sbuf: scratch of 4*S doubles each. */
static void lane_backward_closed_form(const double *q, const double *init,
                                      const double *d_cum, double *d_q,
                                      double *d_init, int64_t S, int64_t stride,
                                      double *pbuf, double *sbuf)
{
    if (S == 0) {
        memset(d_init, 0, 4 * sizeof(double));
        return;
    }
    double P[4] = {1.0, 0.0, 0.0, 0.0}, tmp[4];
    for (int64_t t = 0; t < S; ++t) {
        hamilton(q + 4 * t * stride, P, tmp);
        memcpy(P, tmp, sizeof P);
        memcpy(pbuf + 4 * t, P, sizeof P);
    }
    /* Reverse cumulative sum of conj(P_s) (x) d_cum[s]. */
    double acc[4] = {0.0, 0.0, 0.0, 0.0};
    for (int64_t t = S - 1; t >= 0; --t) {
        double cp[4], term[4];
        conjugate(pbuf + 4 * t, cp);
        hamilton(cp, d_cum + 4 * t * stride, term);
        for (int k = 0; k < 4; ++k) acc[k] += term[k];
        memcpy(sbuf + 4 * t, acc, sizeof acc);
    }
    for (int64_t t = 0; t < S; ++t) {
        double G[4], prev[4], cprev[4];
        hamilton(pbuf + 4 * t, sbuf + 4 * t, G);
        if (t == 0) {
            memcpy(prev, init, sizeof prev);
        } else {
            hamilton(pbuf + 4 * (t - 1), init, prev);   /* cum[t-1] = P_{t-1} (x) init */
        }
        conjugate(prev, cprev);
        hamilton(G, cprev, d_q + 4 * t * stride);
    }
    memcpy(d_init, sbuf, 4 * sizeof(double));
}

/* ---------------------------------------------------------------------------
 * Threading over lanes.
 * ------------------------------------------------------------------------- */

enum { JOB_FWD = 0, JOB_BWD = 1, JOB_BWD_CLOSED = 2 };

typedef struct {
    int kind;
    const double *q, *init, *d_cum;
    double *cum, *d_q, *d_init;
    int64_t B, S, HJ;
    int64_t lane_begin, lane_end;
    int status;
} job_t;

static void *run_job(void *arg)
{
    job_t *jb = (job_t *)arg;
    const int64_t S = jb->S, HJ = jb->HJ;
    double *buf0 = NULL, *buf1 = NULL;
    if (jb->kind != JOB_FWD && S > 0) {
        buf0 = (double *)malloc((size_t)S * 4 * sizeof(double));
        if (jb->kind == JOB_BWD_CLOSED)
            buf1 = (double *)malloc((size_t)S * 4 * sizeof(double));
        if (!buf0 || (jb->kind == JOB_BWD_CLOSED && !buf1)) {
            free(buf0);
            free(buf1);
            jb->status = -2;
            return NULL;
        }
    }
    for (int64_t lane = jb->lane_begin; lane < jb->lane_end; ++lane) {
        const int64_t b = lane / HJ, hj = lane % HJ;
        const int64_t base = (b * S * HJ + hj) * 4;   /* element (b, 0, hj) */
        const double *init = jb->init + 4 * lane;
        if (jb->kind == JOB_FWD) {
            lane_forward(jb->q + base, init, jb->cum + base, S, HJ);
        } else if (jb->kind == JOB_BWD) {
            lane_backward_recurrence(jb->q + base, init, jb->d_cum + base,
                                     jb->d_q + base, jb->d_init + 4 * lane, S,
                                     HJ, buf0);
        } else {
            lane_backward_closed_form(jb->q + base, init, jb->d_cum + base,
                                      jb->d_q + base, jb->d_init + 4 * lane, S,
                                      HJ, buf0, buf1);
        }
    }
    free(buf0);
    free(buf1);
    jb->status = 0;
    return NULL;
}

static int run_lanes(job_t proto, int nthreads)
{
    if (proto.B < 0 || proto.S < 0 || proto.HJ < 0) return -1;
    const int64_t lanes = proto.B * proto.HJ;
    if (lanes == 0) return 0;
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = (n > 0) ? (int)n : 1;
    }
    if (nthreads > lanes) nthreads = (int)lanes;
    if (nthreads > 1024) nthreads = 1024;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int status = 0;
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = proto;
        jobs[i].lane_begin = lanes * i / nthreads;
        jobs[i].lane_end = lanes * (i + 1) / nthreads;
        jobs[i].status = 0;
        if (nthreads == 1 || pthread_create(&tids[i], NULL, run_job, &jobs[i]) != 0) {
            run_job(&jobs[i]);   /* single thread, or thread creation failed */
            tids[i] = 0;
        } else {
            ++started;
        }
    }
    for (int i = 0; i < nthreads; ++i) {
        if (tids[i]) pthread_join(tids[i], NULL);
        if (jobs[i].status != 0) status = jobs[i].status;
    }
    (void)started;
    free(jobs);
    free(tids);
    return status;
}

static int check_ptrs(int64_t n, const void *a, const void *b, const void *c)
{
    if (n == 0) return 0;
    return (a && b && c) ? 0 : -1;
}

/* cum[b,t,h,j] = q[b,t,h,j] (x) cum[b,t-1,h,j], cum[b,-1,h,j] = init[b,h,j]. */
int oracle_fwd(const double *q, const double *init, double *cum, int64_t B,
               int64_t S, int64_t H, int64_t J, int nthreads)
{
    if (B < 0 || S < 0 || H < 0 || J < 0) return -1;
    if (check_ptrs(B * S * H * J, q, init, cum)) return -1;
    job_t p;
    memset(&p, 0, sizeof p);
    p.kind = JOB_FWD;
    p.q = q;
    p.init = init;
    p.cum = cum;
    p.B = B;
    p.S = S;
    p.HJ = H * J;
    return run_lanes(p, nthreads);
}

/* Literal reverse recurrence: (q, init, d_cum) -> (d_q, d_init). */
int oracle_bwd(const double *q, const double *init, const double *d_cum,
               double *d_q, double *d_init, int64_t B, int64_t S, int64_t H,
               int64_t J, int nthreads)
{
    if (B < 0 || S < 0 || H < 0 || J < 0) return -1;
    if (check_ptrs(B * H * J, init, d_init, init)) return -1;
    if (check_ptrs(B * S * H * J, q, d_cum, d_q)) return -1;
    job_t p;
    memset(&p, 0, sizeof p);
    p.kind = JOB_BWD;
    p.q = q;
    p.init = init;
    p.d_cum = d_cum;
    p.d_q = d_q;
    p.d_init = d_init;
    p.B = B;
    p.S = S;
    p.HJ = H * J;
    return run_lanes(p, nthreads);
}

/* The page's closed form (prefix product, suffix sum, G = P (x) S). */
int oracle_bwd_closed_form(const double *q, const double *init,
                           const double *d_cum, double *d_q, double *d_init,
                           int64_t B, int64_t S, int64_t H, int64_t J,
                           int nthreads)
{
    if (B < 0 || S < 0 || H < 0 || J < 0) return -1;
    if (check_ptrs(B * H * J, init, d_init, init)) return -1;
    if (check_ptrs(B * S * H * J, q, d_cum, d_q)) return -1;
    job_t p;
    memset(&p, 0, sizeof p);
    p.kind = JOB_BWD_CLOSED;
    p.q = q;
    p.init = init;
    p.d_cum = d_cum;
    p.d_q = d_q;
    p.d_init = d_init;
    p.B = B;
    p.S = S;
    p.HJ = H * J;
    return run_lanes(p, nthreads);
}
