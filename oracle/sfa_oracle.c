/*
 * sfa_oracle.c -- CPU oracle for depth-staggered Fibonacci sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, fp64 statement of
 * what the GPU path computes.  Only the tests, the package smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA library, and neither side includes the other.
 *
 * Source of every rule below: "Depth-Staggered Fibonacci Spacing for Sparse
 * Attention: Static Schedules Beat Learned Dilation and Extrapolate Where Dense
 * Attention Fails" (arXiv 2606.28560), section 2 "Method":
 *   - "Attended set": query i attends the dense window of distances 0..W
 *     (self included) plus one rung per base offset f_k at the continuous
 *     distance d_k = alpha * f_k; each rung reads the key/value row at i - d_k by
 *     linear interpolation of the rows at the whole distances just below and
 *     just above d_k; RoPE is
 *     applied at the true positions before the gather; the offset set is the
 *     same for every query.
 *   - "Per-layer scalar": alpha = 0.5 + sigmoid(theta), theta the only added
 *     parameter.
 *   - "Implementation notes": the interpolated gather exists so that alpha
 *     receives a gradient even at integer positions.
 * Section 3 "Model and training" fixes the attention shape used here (8 query
 * heads, 2 key/value heads, head dimension 64, RoPE theta 1e4).
 *
 * Readings where the paper is silent (each one is also listed in the design
 * notes of the repository):
 *   - the softmax scale is a parameter (1/sqrt(64) = 1/8 in every workload);
 *   - a rung whose distance satisfies d_k <= W is dropped (it lies inside the
 *     window already);
 *   - a rung is masked for query i when i - ceil(d_k) < 0 (no clamping, no zero
 *     rows); at an integer distance (t = 0) that is i - d_k < 0;
 *   - the interpolation puts weight (1 - t) on row i - floor(d_k) and weight t on
 *     row i - floor(d_k) - 1, t = d_k - floor(d_k), for keys and values alike;
 *   - d_k is the fp32 product of fp32(alpha) and fp32(f_k), rounded to nearest,
 *     when cfg.d_fp32 is set (the GPU path uses the same rule, so floor and
 *     ceil never disagree); with d_fp32 = 0 it is the fp64 product (used by the
 *     finite-difference tests, which need a smooth map alpha -> d_k);
 *   - RoPE pairs dimension m with m + D/2 ("rotate half"), angle pos *
 *     rope_theta^(-2m/D); rope_theta <= 0 means no rotation;
 *   - query head h reads key/value head h / (Hq/Hkv);
 *   - the derivative of floor/ceil and of the drop/mask decisions is zero, and
 *     at t = 0 the t-derivative of an entry whose far row (distance n + 1) lies before the
 *     sequence start is zero (that row does not exist).
 *
 * Layout of every tensor: row-major [B][T][H][D], D fastest, fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, T, Hq, Hkv, D;   /* shapes */
    int W;                  /* window covers distances 0..W */
    int K;                  /* number of base offsets */
    const double *f;        /* base offsets f_k, K values */
    double alpha;           /* the layer's scalar */
    int d_fp32;             /* 1: d_k = fl32(fl32(alpha) * fl32(f_k)); 0: fp64 product */
    double rope_theta;      /* <= 0: inputs are used as they are */
    double scale;           /* softmax scale */
    int nthreads;           /* worker threads (>= 1) */
    int round_offsets;      /* 1: every distance rounded to the nearest integer */
} oracle_cfg;

/* One attended key: the score and the value read are
 *   wa * row ra + wb * row rb   (row rb unused when wb == 0 or rb < 0).
 * rung < 0 marks a window entry. */
typedef struct {
    double wa, wb;
    int ra, rb;
    int rung;
} entry;

/* ---------------------------------------------------------------- rungs -- */

/* Distance of rung k ("Attended set": d_k = alpha * f_k).  With
 * round_offsets the distance is the nearest integer, halves rounded up (the
 * static schedules "with integer offsets" of "Implementation notes"). */
static double rung_distance(const oracle_cfg *c, int k)
{
    double d;
    if (c->d_fp32) {
        volatile float a = (float)c->alpha;
        volatile float fk = (float)c->f[k];
        volatile float df = a * fk;       /* one fp32 multiply, round to nearest */
        d = (double)df;
    } else {
        d = c->alpha * c->f[k];
    }
    return c->round_offsets ? floor(d + 0.5) : d;
}

/* The explicit key list of query i ("Attended set").  Returns the count. */
static int build_entries(const oracle_cfg *c, int i, entry *e)
{
    int n = 0;
    for (int delta = 0; delta <= c->W; ++delta) {
        if (i - delta < 0)
            break;
        e[n].wa = 1.0; e[n].wb = 0.0;
        e[n].ra = i - delta; e[n].rb = -1;
        e[n].rung = -1;
        ++n;
    }
    for (int k = 0; k < c->K; ++k) {
        double d = rung_distance(c, k);
        if (d <= (double)c->W)
            continue;                     /* inside the window already: dropped */
        double fl = floor(d), ce = ceil(d), t = d - fl;
        if ((double)i - ce < 0.0)
            continue;                     /* reaches before the sequence start */
        int a = i - (int)fl;
        e[n].wa = 1.0 - t;
        e[n].wb = t;
        e[n].ra = a;
        e[n].rb = (a - 1 >= 0) ? a - 1 : -1;
        e[n].rung = k;
        ++n;
    }
    return n;
}

int oracle_max_entries(const oracle_cfg *c) { return c->W + 1 + c->K; }

/* ----------------------------------------------------------------- RoPE -- */

/* y = R(pos) x, rotate-half pairing (m, m + D/2), angle pos * theta^(-2m/D).
 * inverse != 0 applies R(pos)^T instead. */
static void rope_vec(const double *x, double *y, int D, int pos, double theta, int inverse)
{
    int h = D / 2;
    if (theta <= 0.0) {
        memmove(y, x, sizeof(double) * (size_t)D);
        return;
    }
    for (int m = 0; m < h; ++m) {
        double w = pow(theta, -2.0 * (double)m / (double)D);
        double ang = (double)pos * w;
        double cs = cos(ang), sn = sin(ang);
        double x0 = x[m], x1 = x[m + h];
        if (!inverse) {
            y[m] = x0 * cs - x1 * sn;
            y[m + h] = x1 * cs + x0 * sn;
        } else {
            y[m] = x0 * cs + x1 * sn;
            y[m + h] = x1 * cs - x0 * sn;
        }
    }
}

/* Rotate a whole [B][T][H][D] tensor at its true positions (exported so the
 * tests can hand rotated inputs to a library attention routine). */
void oracle_rope(int B, int T, int H, int D, double theta, int inverse,
                 const double *x, double *y)
{
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t)
            for (int hh = 0; hh < H; ++hh) {
                size_t off = (((size_t)b * T + t) * H + hh) * (size_t)D;
                rope_vec(x + off, y + off, D, t, theta, inverse);
            }
}

static size_t idx(const oracle_cfg *c, int H, int b, int t, int h)
{
    return (((size_t)b * c->T + t) * H + h) * (size_t)c->D;
}

static double dot(const double *a, const double *b, int D)
{
    double s = 0.0;
    for (int d = 0; d < D; ++d)
        s += a[d] * b[d];
    return s;
}

/* ------------------------------------------------------------- threading -- */

typedef struct {
    const oracle_cfg *c;
    const double *q, *k, *v, *dO;
    const double *khat;      /* rotated keys [B][T][Hkv][D] */
    double *o, *lse;         /* forward outputs (may be NULL in backward) */
    double *dq, *dkhat, *dv; /* backward accumulators */
    double *dt;              /* [B][K] per-sequence dL/dt_k */
    const int *rows;         /* sampled (b, i) pairs or NULL */
    int nrows;
    int lo, hi;              /* work range */
    int status;
} job;

static int run_jobs(const oracle_cfg *c, job *proto, int nwork, void *(*fn)(void *))
{
    int nt = c->nthreads < 1 ? 1 : c->nthreads;
    if (nt > nwork)
        nt = nwork < 1 ? 1 : nwork;
    job *jobs = (job *)calloc((size_t)nt, sizeof(job));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th);
        return -1;
    }
    int status = 0;
    for (int w = 0; w < nt; ++w) {
        jobs[w] = *proto;
        jobs[w].lo = (int)((long long)nwork * w / nt);
        jobs[w].hi = (int)((long long)nwork * (w + 1) / nt);
        jobs[w].status = 0;
    }
    if (nt == 1) {
        fn(&jobs[0]);
    } else {
        for (int w = 0; w < nt; ++w)
            pthread_create(&th[w], NULL, fn, &jobs[w]);
        for (int w = 0; w < nt; ++w)
            pthread_join(th[w], NULL);
    }
    for (int w = 0; w < nt; ++w)
        if (jobs[w].status)
            status = jobs[w].status;
    free(jobs); free(th);
    return status;
}

static double *rotate_keys(const oracle_cfg *c, const double *k)
{
    size_t n = (size_t)c->B * c->T * c->Hkv * c->D;
    double *kh = (double *)malloc(sizeof(double) * (n ? n : 1));
    if (kh)
        oracle_rope(c->B, c->T, c->Hkv, c->D, c->rope_theta, 0, k, kh);
    return kh;
}

/* --------------------------------------------------------------- forward -- */

/* Attention of one query row (b, i) over its key list, every query head.
 * Softmax over the union set of window and rung entries (the "Attended set"). */
static int forward_row(const job *J, int b, int i, double *o_out, double *lse_out)
{
    const oracle_cfg *c = J->c;
    int D = c->D, G = c->Hq / c->Hkv;
    int ne_max = oracle_max_entries(c);
    entry *e = (entry *)malloc(sizeof(entry) * (size_t)ne_max);
    double *s = (double *)malloc(sizeof(double) * (size_t)ne_max);
    double *qh = (double *)malloc(sizeof(double) * (size_t)D);
    double *kt = (double *)malloc(sizeof(double) * (size_t)D);
    if (!e || !s || !qh || !kt) {
        free(e); free(s); free(qh); free(kt);
        return -1;
    }
    int ne = build_entries(c, i, e);
    for (int h = 0; h < c->Hq; ++h) {
        int g = h / G;
        rope_vec(J->q + idx(c, c->Hq, b, i, h), qh, D, i, c->rope_theta, 0);
        double m = -INFINITY;
        for (int n = 0; n < ne; ++n) {
            const double *ka = J->khat + idx(c, c->Hkv, b, e[n].ra, g);
            for (int d = 0; d < D; ++d)
                kt[d] = e[n].wa * ka[d];
            if (e[n].wb != 0.0) {
                const double *kb = J->khat + idx(c, c->Hkv, b, e[n].rb, g);
                for (int d = 0; d < D; ++d)
                    kt[d] += e[n].wb * kb[d];
            }
            s[n] = c->scale * dot(qh, kt, D);
            if (s[n] > m)
                m = s[n];
        }
        double l = 0.0;
        for (int n = 0; n < ne; ++n)
            l += exp(s[n] - m);
        double *o = o_out + (size_t)h * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int n = 0; n < ne; ++n) {
            double p = exp(s[n] - m) / l;
            const double *va = J->v + idx(c, c->Hkv, b, e[n].ra, g);
            for (int d = 0; d < D; ++d)
                o[d] += p * e[n].wa * va[d];
            if (e[n].wb != 0.0) {
                const double *vb = J->v + idx(c, c->Hkv, b, e[n].rb, g);
                for (int d = 0; d < D; ++d)
                    o[d] += p * e[n].wb * vb[d];
            }
        }
        if (lse_out)
            lse_out[h] = m + log(l);
    }
    free(e); free(s); free(qh); free(kt);
    return 0;
}

static void *forward_worker(void *arg)
{
    job *J = (job *)arg;
    const oracle_cfg *c = J->c;
    for (int w = J->lo; w < J->hi; ++w) {
        int b, i;
        if (J->rows) {
            b = J->rows[2 * w];
            i = J->rows[2 * w + 1];
        } else {
            b = w / c->T;
            i = w % c->T;
        }
        double *o = J->o + (size_t)w * c->Hq * c->D;
        double *lse = J->lse ? J->lse + (size_t)w * c->Hq : NULL;
        if (forward_row(J, b, i, o, lse)) {
            J->status = -1;
            return NULL;
        }
    }
    return NULL;
}

static int check_cfg(const oracle_cfg *c)
{
    if (c->B < 0 || c->T < 0 || c->Hq <= 0 || c->Hkv <= 0 || c->D <= 0 || (c->D & 1))
        return -2;
    if (c->Hq % c->Hkv || c->W < 0 || c->K < 0 || (c->K > 0 && !c->f))
        return -2;
    return 0;
}

/* Full forward: o [B][T][Hq][D], lse [B][T][Hq] (lse may be NULL). */
int oracle_forward(const oracle_cfg *c, const double *q, const double *k, const double *v,
                   double *o, double *lse)
{
    int st = check_cfg(c);
    if (st)
        return st;
    if (c->B == 0 || c->T == 0)
        return 0;
    double *kh = rotate_keys(c, k);
    if (!kh)
        return -1;
    job J;
    memset(&J, 0, sizeof J);
    J.c = c; J.q = q; J.k = k; J.v = v; J.khat = kh; J.o = o; J.lse = lse;
    st = run_jobs(c, &J, c->B * c->T, forward_worker);
    free(kh);
    return st;
}

/* Forward of sampled query rows only: rows = nrows pairs (b, i); o is
 * [nrows][Hq][D], lse [nrows][Hq] (may be NULL).  Each row is computed from
 * scratch exactly as in oracle_forward. */
int oracle_forward_rows(const oracle_cfg *c, const double *q, const double *k, const double *v,
                        int nrows, const int *rows, double *o, double *lse)
{
    int st = check_cfg(c);
    if (st)
        return st;
    for (int r = 0; r < nrows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= c->B || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= c->T)
            return -2;
    if (nrows == 0)
        return 0;
    double *kh = rotate_keys(c, k);
    if (!kh)
        return -1;
    job J;
    memset(&J, 0, sizeof J);
    J.c = c; J.q = q; J.k = k; J.v = v; J.khat = kh; J.o = o; J.lse = lse;
    J.rows = rows; J.nrows = nrows;
    st = run_jobs(c, &J, nrows, forward_worker);
    free(kh);
    return st;
}

/* -------------------------------------------------------------- backward -- */

/* Gradients of L = sum(dO * O) for one sequence b.  Per query row and head
 * (g = h / G), with s_e = scale * qhat . ktilde_e, p = softmax(s),
 * Dh = dO . o:
 *   dp_e = dO . vtilde_e,  ds_e = p_e (dp_e - Dh)
 *   dqhat += scale * ds_e * ktilde_e
 *   dkhat[ra] += wa * scale * ds_e * qhat,  dkhat[rb] += wb * (same)
 *   dv[ra] += wa * p_e * dO,                dv[rb] += wb * (same)
 *   dL/dt_k += scale * ds_e * qhat . (khat[rb] - khat[ra]) + p_e * dO . (v[rb] - v[ra])
 * ("Implementation notes": the interpolation weight t carries the gradient to
 * alpha).  Rotations are undone at the end: dq = R(i)^T dqhat,
 * dk = R(j)^T dkhat. */
static void *backward_worker(void *arg)
{
    job *J = (job *)arg;
    const oracle_cfg *c = J->c;
    int D = c->D, G = c->Hq / c->Hkv;
    int ne_max = oracle_max_entries(c);
    entry *e = (entry *)malloc(sizeof(entry) * (size_t)ne_max);
    double *s = (double *)malloc(sizeof(double) * (size_t)ne_max);
    double *p = (double *)malloc(sizeof(double) * (size_t)ne_max);
    double *qh = (double *)malloc(sizeof(double) * (size_t)D);
    double *kt = (double *)malloc(sizeof(double) * (size_t)D);
    double *vt = (double *)malloc(sizeof(double) * (size_t)D);
    double *o = (double *)malloc(sizeof(double) * (size_t)D);
    double *dqh = (double *)malloc(sizeof(double) * (size_t)D);
    if (!e || !s || !p || !qh || !kt || !vt || !o || !dqh) {
        J->status = -1;
        goto out;
    }
    for (int b = J->lo; b < J->hi; ++b) {
        double *dt = J->dt + (size_t)b * (c->K > 0 ? c->K : 1);
        for (int i = 0; i < c->T; ++i) {
            int ne = build_entries(c, i, e);
            for (int h = 0; h < c->Hq; ++h) {
                int g = h / G;
                const double *dO = J->dO + idx(c, c->Hq, b, i, h);
                rope_vec(J->q + idx(c, c->Hq, b, i, h), qh, D, i, c->rope_theta, 0);
                /* recompute the forward of this row */
                double m = -INFINITY;
                for (int n = 0; n < ne; ++n) {
                    const double *ka = J->khat + idx(c, c->Hkv, b, e[n].ra, g);
                    for (int d = 0; d < D; ++d)
                        kt[d] = e[n].wa * ka[d];
                    if (e[n].wb != 0.0) {
                        const double *kb = J->khat + idx(c, c->Hkv, b, e[n].rb, g);
                        for (int d = 0; d < D; ++d)
                            kt[d] += e[n].wb * kb[d];
                    }
                    s[n] = c->scale * dot(qh, kt, D);
                    if (s[n] > m)
                        m = s[n];
                }
                double l = 0.0;
                for (int n = 0; n < ne; ++n)
                    l += exp(s[n] - m);
                for (int d = 0; d < D; ++d)
                    o[d] = 0.0;
                for (int n = 0; n < ne; ++n) {
                    p[n] = exp(s[n] - m) / l;
                    const double *va = J->v + idx(c, c->Hkv, b, e[n].ra, g);
                    for (int d = 0; d < D; ++d)
                        vt[d] = e[n].wa * va[d];
                    if (e[n].wb != 0.0) {
                        const double *vb = J->v + idx(c, c->Hkv, b, e[n].rb, g);
                        for (int d = 0; d < D; ++d)
                            vt[d] += e[n].wb * vb[d];
                    }
                    for (int d = 0; d < D; ++d)
                        o[d] += p[n] * vt[d];
                }
                double Dh = dot(dO, o, D);
                for (int d = 0; d < D; ++d)
                    dqh[d] = 0.0;
                for (int n = 0; n < ne; ++n) {
                    const double *ka = J->khat + idx(c, c->Hkv, b, e[n].ra, g);
                    const double *va = J->v + idx(c, c->Hkv, b, e[n].ra, g);
                    const double *kb = e[n].rb >= 0 ? J->khat + idx(c, c->Hkv, b, e[n].rb, g) : NULL;
                    const double *vb = e[n].rb >= 0 ? J->v + idx(c, c->Hkv, b, e[n].rb, g) : NULL;
                    for (int d = 0; d < D; ++d) {
                        kt[d] = e[n].wa * ka[d];
                        vt[d] = e[n].wa * va[d];
                    }
                    if (e[n].wb != 0.0)
                        for (int d = 0; d < D; ++d) {
                            kt[d] += e[n].wb * kb[d];
                            vt[d] += e[n].wb * vb[d];
                        }
                    double dp = dot(dO, vt, D);
                    double ds = p[n] * (dp - Dh);
                    for (int d = 0; d < D; ++d)
                        dqh[d] += c->scale * ds * kt[d];
                    double *dka = J->dkhat + idx(c, c->Hkv, b, e[n].ra, g);
                    double *dva = J->dv + idx(c, c->Hkv, b, e[n].ra, g);
                    for (int d = 0; d < D; ++d) {
                        dka[d] += e[n].wa * c->scale * ds * qh[d];
                        dva[d] += e[n].wa * p[n] * dO[d];
                    }
                    if (e[n].wb != 0.0) {
                        double *dkb = J->dkhat + idx(c, c->Hkv, b, e[n].rb, g);
                        double *dvb = J->dv + idx(c, c->Hkv, b, e[n].rb, g);
                        for (int d = 0; d < D; ++d) {
                            dkb[d] += e[n].wb * c->scale * ds * qh[d];
                            dvb[d] += e[n].wb * p[n] * dO[d];
                        }
                    }
                    if (e[n].rung >= 0 && e[n].rb >= 0) {
                        double gk = 0.0, gv = 0.0;
                        for (int d = 0; d < D; ++d) {
                            gk += qh[d] * (kb[d] - ka[d]);
                            gv += dO[d] * (vb[d] - va[d]);
                        }
                        dt[e[n].rung] += c->scale * ds * gk + p[n] * gv;
                    }
                }
                rope_vec(dqh, J->dq + idx(c, c->Hq, b, i, h), D, i, c->rope_theta, 1);
            }
        }
    }
out:
    free(e); free(s); free(p); free(qh); free(kt); free(vt); free(o); free(dqh);
    return NULL;
}

/* Full backward of L = sum(dO * O).  Outputs dq [B][T][Hq][D], dk and dv
 * [B][T][Hkv][D], dalpha = sum_k f_k dL/dt_k (since d d_k / d alpha = f_k), and
 * dtheta = dalpha * (alpha - 0.5)(1.5 - alpha), the derivative of
 * alpha = 0.5 + sigmoid(theta) ("Per-layer scalar").  dt (may be NULL) receives
 * the K summed dL/dt_k. */
int oracle_backward(const oracle_cfg *c, const double *q, const double *k, const double *v,
                    const double *dO, double *dq, double *dk, double *dv,
                    double *dalpha, double *dtheta, double *dt_out)
{
    int st = check_cfg(c);
    if (st)
        return st;
    size_t nkv = (size_t)c->B * c->T * c->Hkv * c->D;
    size_t nq = (size_t)c->B * c->T * c->Hq * c->D;
    memset(dq, 0, sizeof(double) * nq);
    memset(dv, 0, sizeof(double) * nkv);
    int Kc = c->K > 0 ? c->K : 1;
    double *dt = (double *)calloc((size_t)(c->B > 0 ? c->B : 1) * Kc, sizeof(double));
    double *kh = rotate_keys(c, k);
    double *dkh = (double *)calloc(nkv ? nkv : 1, sizeof(double));
    if (!dt || !kh || !dkh) {
        free(dt); free(kh); free(dkh);
        return -1;
    }
    job J;
    memset(&J, 0, sizeof J);
    J.c = c; J.q = q; J.k = k; J.v = v; J.dO = dO; J.khat = kh;
    J.dq = dq; J.dkhat = dkh; J.dv = dv; J.dt = dt;
    st = (c->B > 0 && c->T > 0) ? run_jobs(c, &J, c->B, backward_worker) : 0;
    if (!st) {
        oracle_rope(c->B, c->T, c->Hkv, c->D, c->rope_theta, 1, dkh, dk);
        double da = 0.0;
        for (int kk = 0; kk < c->K; ++kk) {
            double tot = 0.0;
            for (int b = 0; b < c->B; ++b)
                tot += dt[(size_t)b * Kc + kk];
            if (dt_out)
                dt_out[kk] = tot;
            /* d d_k / d alpha: f_k, or 0 once the distance is rounded */
            da += (c->round_offsets ? 0.0 : c->f[kk]) * tot;
        }
        *dalpha = da;
        *dtheta = da * (c->alpha - 0.5) * (1.5 - c->alpha);
    }
    free(dt); free(kh); free(dkh);
    return st;
}
