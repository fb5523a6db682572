/*
 * conv_ref.c -- fp64 CPU oracle for the small-spatial, large-batch conv2d layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * What it computes (PufferLib PR #522, "Speedups to gemm_conv_forward and
 * gemm_conv_backward kernels": the layer-1 / layer-2 bench blocks, which name
 * the three results "forward", "backward wgrad" and "backward d_input", and
 * print the shapes 11x15 K=5 S=3 -> 3x4 relu=1 and 3x4 K=3 S=1 -> 1x2 relu=0):
 *
 *   OH = floor((H - K) / S) + 1,  OW = floor((W - K) / S) + 1  (no padding;
 *   the printed 11x15 -> 3x4 only holds with the floor).
 *
 *   forward   y[b,oc,oh,ow]  = act( sum_{ic,kh,kw} x[b,ic,oh*S+kh,ow*S+kw] * w[oc,ic,kh,kw] )
 *             act = max(., 0) when relu, identity otherwise.
 *
 *   g         = dy * [y > 0] when relu (y is the forward output the caller
 *               holds), g = dy otherwise.
 *
 *   d_input   dx[b,ic,h,w]   = sum over (oc, kh, kw, oh, ow) with oh*S+kh = h and
 *                              ow*S+kw = w of g[b,oc,oh,ow] * w[oc,ic,kh,kw]
 *   wgrad     dw[oc,ic,kh,kw] = sum_{b,oh,ow} g[b,oc,oh,ow] * x[b,ic,oh*S+kh,ow*S+kw]
 *
 * The layer's bias (the same PR's "n3_conv_bias_grad" bench blocks time the
 * gradient of a per-output-channel conv bias, conv1: OC=128 x 12 positions,
 * conv2: OC=128 x 2): the bias is added to the sum before the activation,
 *
 *   forward+bias  y[b,oc,oh,ow] = act( bias[oc] + sum_{ic,kh,kw} ... as above )
 *   bias grad     db[oc]        = sum_{b,oh,ow} g[b,oc,oh,ow]
 *
 * Each output is accumulated in fp64 by direct loops in a fixed order, and
 * its "denominator" D = sum of |term| over the same terms is returned beside
 * it, so that a caller can form the normalised error |out - ref| / D.
 *
 * Layouts: x, dx NCHW (B,IC,H,W); y, dy, g (B,OC,OH,OW); w, dw (OC,IC,K,K);
 * all arrays dense, row-major, double.
 *
 * Threads: every output element is computed start-to-finish by one thread
 * in the same order, so results do not depend on the thread count.
 *
 * Parity pins: brute force against an independent im2col-matrix formulation
 * (with the bias as an extra row of ones), the 1x1/stride-1 matmul special
 * case, the delta-input case, the zero-weight case (y = act(bias)), the
 * adjoint identity, central finite differences (in x, w and the bias) and the
 * printed output sizes (tests in tests/test_oracle.py).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    int64_t B, IC, OC, H, W, K, S;
    int32_t relu;
} ref_shape_t;

static int64_t ref_out_dim(int64_t n, int64_t K, int64_t S) { return (n - K) / S + 1; }

/* Output size of one spatial axis, exported so tests can pin it. */
int64_t oracle_out_dim(int64_t n, int64_t K, int64_t S) { return ref_out_dim(n, K, S); }

/* g = dy masked by the forward output when relu is set. */
static double ref_g(const ref_shape_t* s, const double* dy, const double* y, int64_t i)
{
    if (s->relu && !(y[i] > 0.0)) return 0.0;
    return dy[i];
}

typedef struct {
    const ref_shape_t* s;
    const double *a, *b, *c; /* operation-specific inputs */
    double *out, *den;
    int64_t lo, hi;          /* range of the outermost loop index */
} ref_job_t;

/* ---- forward: outer index b; j->c is the bias (OC) or NULL ---------------- */
static void* ref_fwd_range(void* arg)
{
    const ref_job_t* j = (const ref_job_t*)arg;
    const ref_shape_t* s = j->s;
    const double* x = j->a;
    const double* w = j->b;
    const int64_t OH = ref_out_dim(s->H, s->K, s->S), OW = ref_out_dim(s->W, s->K, s->S);
    for (int64_t b = j->lo; b < j->hi; ++b)
        for (int64_t oc = 0; oc < s->OC; ++oc)
            for (int64_t oh = 0; oh < OH; ++oh)
                for (int64_t ow = 0; ow < OW; ++ow) {
                    double acc = 0.0, den = 0.0;
                    for (int64_t ic = 0; ic < s->IC; ++ic)
                        for (int64_t kh = 0; kh < s->K; ++kh)
                            for (int64_t kw = 0; kw < s->K; ++kw) {
                                const int64_t h = oh * s->S + kh, ww = ow * s->S + kw;
                                const double t = x[((b * s->IC + ic) * s->H + h) * s->W + ww] *
                                                 w[((oc * s->IC + ic) * s->K + kh) * s->K + kw];
                                acc += t;
                                den += fabs(t);
                            }
                    if (j->c) { /* bias, added to the finished sum */
                        const double bv = j->c[oc];
                        acc += bv;
                        den += fabs(bv);
                    }
                    const int64_t o = ((b * s->OC + oc) * OH + oh) * OW + ow;
                    j->out[o] = (s->relu && !(acc > 0.0)) ? 0.0 : acc;
                    if (j->den) j->den[o] = den;
                }
    return NULL;
}

/* ---- d_input: outer index b; gather form of the sum ----------------------- */
static void* ref_dgrad_range(void* arg)
{
    const ref_job_t* j = (const ref_job_t*)arg;
    const ref_shape_t* s = j->s;
    const double* dy = j->a;
    const double* w = j->b;
    const double* y = j->c;
    const int64_t OH = ref_out_dim(s->H, s->K, s->S), OW = ref_out_dim(s->W, s->K, s->S);
    for (int64_t b = j->lo; b < j->hi; ++b)
        for (int64_t ic = 0; ic < s->IC; ++ic)
            for (int64_t h = 0; h < s->H; ++h)
                for (int64_t ww = 0; ww < s->W; ++ww) {
                    double acc = 0.0, den = 0.0;
                    for (int64_t oc = 0; oc < s->OC; ++oc)
                        for (int64_t kh = 0; kh < s->K; ++kh) {
                            const int64_t th = h - kh; /* = oh*S when the row is touched */
                            if (th < 0 || th % s->S != 0 || th / s->S >= OH) continue;
                            const int64_t oh = th / s->S;
                            for (int64_t kw = 0; kw < s->K; ++kw) {
                                const int64_t tw = ww - kw;
                                if (tw < 0 || tw % s->S != 0 || tw / s->S >= OW) continue;
                                const int64_t ow = tw / s->S;
                                const double t =
                                    ref_g(s, dy, y, ((b * s->OC + oc) * OH + oh) * OW + ow) *
                                    w[((oc * s->IC + ic) * s->K + kh) * s->K + kw];
                                acc += t;
                                den += fabs(t);
                            }
                        }
                    const int64_t o = ((b * s->IC + ic) * s->H + h) * s->W + ww;
                    j->out[o] = acc;
                    if (j->den) j->den[o] = den;
                }
    return NULL;
}

/* ---- wgrad: outer index oc ------------------------------------------------ */
static void* ref_wgrad_range(void* arg)
{
    const ref_job_t* j = (const ref_job_t*)arg;
    const ref_shape_t* s = j->s;
    const double* x = j->a;
    const double* dy = j->b;
    const double* y = j->c;
    const int64_t OH = ref_out_dim(s->H, s->K, s->S), OW = ref_out_dim(s->W, s->K, s->S);
    for (int64_t oc = j->lo; oc < j->hi; ++oc)
        for (int64_t ic = 0; ic < s->IC; ++ic)
            for (int64_t kh = 0; kh < s->K; ++kh)
                for (int64_t kw = 0; kw < s->K; ++kw) {
                    double acc = 0.0, den = 0.0;
                    for (int64_t b = 0; b < s->B; ++b)
                        for (int64_t oh = 0; oh < OH; ++oh)
                            for (int64_t ow = 0; ow < OW; ++ow) {
                                const double t =
                                    ref_g(s, dy, y, ((b * s->OC + oc) * OH + oh) * OW + ow) *
                                    x[((b * s->IC + ic) * s->H + oh * s->S + kh) * s->W +
                                      ow * s->S + kw];
                                acc += t;
                                den += fabs(t);
                            }
                    const int64_t o = ((oc * s->IC + ic) * s->K + kh) * s->K + kw;
                    j->out[o] = acc;
                    if (j->den) j->den[o] = den;
                }
    return NULL;
}

/* ---- bias grad: outer index oc -------------------------------------------- */
static void* ref_bgrad_range(void* arg)
{
    const ref_job_t* j = (const ref_job_t*)arg;
    const ref_shape_t* s = j->s;
    const double* dy = j->a;
    const double* y = j->c;
    const int64_t OH = ref_out_dim(s->H, s->K, s->S), OW = ref_out_dim(s->W, s->K, s->S);
    for (int64_t oc = j->lo; oc < j->hi; ++oc) {
        double acc = 0.0, den = 0.0;
        for (int64_t b = 0; b < s->B; ++b)
            for (int64_t oh = 0; oh < OH; ++oh)
                for (int64_t ow = 0; ow < OW; ++ow) {
                    const double t = ref_g(s, dy, y, ((b * s->OC + oc) * OH + oh) * OW + ow);
                    acc += t;
                    den += fabs(t);
                }
        j->out[oc] = acc;
        if (j->den) j->den[oc] = den;
    }
    return NULL;
}

/* Split [0, n) into nthreads contiguous ranges and run fn on each. */
static int ref_run(void* (*fn)(void*), ref_job_t proto, int64_t n, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    ref_job_t jobs[256];
    pthread_t tid[256];
    int started[256] = {0};
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].lo = n * t / nthreads;
        jobs[t].hi = n * (t + 1) / nthreads;
    }
    int rc = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, fn, &jobs[t]) == 0)
            started[t] = 1;
        else
            fn(&jobs[t]); /* could not spawn: run the range inline */
    }
    fn(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) rc |= pthread_join(tid[t], NULL);
    return rc;
}

static int ref_valid(const ref_shape_t* s)
{
    return s && s->B >= 0 && s->IC >= 1 && s->OC >= 1 && s->K >= 1 && s->S >= 1 &&
           s->H >= s->K && s->W >= s->K;
}

/* y, den: (B,OC,OH,OW).  den may be NULL.  Returns 0 on success. */
int oracle_conv_fwd(const ref_shape_t* s, const double* x, const double* w, double* y,
                    double* den, int nthreads)
{
    if (!ref_valid(s) || !x || !w || !y) return -1;
    ref_job_t p = {s, x, w, NULL, y, den, 0, 0};
    return ref_run(ref_fwd_range, p, s->B, nthreads);
}

/* dx, den: (B,IC,H,W).  y is required when s->relu, ignored otherwise. */
int oracle_conv_bwd_data(const ref_shape_t* s, const double* dy, const double* w,
                         const double* y, double* dx, double* den, int nthreads)
{
    if (!ref_valid(s) || !dy || !w || !dx || (s->relu && !y)) return -1;
    ref_job_t p = {s, dy, w, y, dx, den, 0, 0};
    return ref_run(ref_dgrad_range, p, s->B, nthreads);
}

/* dw, den: (OC,IC,K,K).  y is required when s->relu, ignored otherwise. */
int oracle_conv_bwd_filter(const ref_shape_t* s, const double* x, const double* dy,
                           const double* y, double* dw, double* den, int nthreads)
{
    if (!ref_valid(s) || !x || !dy || !dw || (s->relu && !y)) return -1;
    ref_job_t p = {s, x, dy, y, dw, den, 0, 0};
    return ref_run(ref_wgrad_range, p, s->OC, nthreads);
}

/* y, den: (B,OC,OH,OW); bias: (OC), required.  den may be NULL. */
int oracle_conv_fwd_bias(const ref_shape_t* s, const double* x, const double* w,
                         const double* bias, double* y, double* den, int nthreads)
{
    if (!ref_valid(s) || !x || !w || !bias || !y) return -1;
    ref_job_t p = {s, x, w, bias, y, den, 0, 0};
    return ref_run(ref_fwd_range, p, s->B, nthreads);
}

/* db, den: (OC).  y is required when s->relu, ignored otherwise. */
int oracle_conv_bwd_bias(const ref_shape_t* s, const double* dy, const double* y, double* db,
                         double* den, int nthreads)
{
    if (!ref_valid(s) || !dy || !db || (s->relu && !y)) return -1;
    ref_job_t p = {s, dy, NULL, y, db, den, 0, 0};
    return ref_run(ref_bgrad_range, p, s->OC, nthreads);
}
