/*
 * oracle.c -- fp64 CPU oracle: plain loop nests of the definitions.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).  Nothing here is blocked, fused
 * or reordered beyond what each definition states; threads only split the
 * outer (n, channel) or sample loop, and every output element is computed by
 * one thread in the definition's own summation order, so results do not
 * depend on the thread count.
 *
 * Built with  gcc -O2 -ffp-contract=off -shared -fPIC -pthread  so that no
 * fused multiply-add changes rounding between machines.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* a minimal parallel-for over [0, n) in fixed chunks                   */
/* ------------------------------------------------------------------ */
typedef void (*range_fn)(void *ctx, int64_t begin, int64_t end);

typedef struct {
    range_fn fn;
    void *ctx;
    int64_t n, chunk;
    atomic_llong next;
} par_t;

static void *par_worker(void *arg) {
    par_t *p = (par_t *)arg;
    for (;;) {
        int64_t b = atomic_fetch_add(&p->next, p->chunk);
        if (b >= p->n) break;
        int64_t e = b + p->chunk < p->n ? b + p->chunk : p->n;
        p->fn(p->ctx, b, e);
    }
    return NULL;
}

static void par_for(int64_t n, int nthreads, int64_t chunk, range_fn fn, void *ctx) {
    if (n <= 0) return;
    if (chunk < 1) chunk = 1;
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > (n + chunk - 1) / chunk) nthreads = (int)((n + chunk - 1) / chunk);
    par_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.n = n;
    p.chunk = chunk;
    atomic_init(&p.next, 0);
    if (nthreads == 1) {
        par_worker(&p);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, par_worker, &p) != 0) break;
        ++started;
    }
    if (started == 0) par_worker(&p);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
}

/* ------------------------------------------------------------------ */
/* output sizes                                                         */
/* ------------------------------------------------------------------ */
static int64_t floor_div(int64_t a, int64_t b) {
    int64_t q = a / b;
    if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
    return q;
}

int64_t oracle_conv_out_len(int64_t L, int k, int s, int p, int d) {
    if (L <= 0 || k <= 0 || s <= 0 || p < 0 || d <= 0) return 0;
    int64_t span = L + 2 * (int64_t)p - (int64_t)d * (k - 1) - 1;
    if (span < 0) return 0;
    return floor_div(span, s) + 1;
}

int64_t oracle_convT_out_len(int64_t L, int k, int s, int p, int d, int op) {
    if (L <= 0 || k <= 0 || s <= 0 || p < 0 || d <= 0 || op < 0) return 0;
    int64_t o = (L - 1) * s - 2 * (int64_t)p + (int64_t)d * (k - 1) + op + 1;
    return o > 0 ? o : 0;
}

/* ------------------------------------------------------------------ */
/* shared problem description                                           */
/* ------------------------------------------------------------------ */
typedef struct {
    const double *x, *w, *b;
    double *y;
    int N, Cin, Cout, G;
    int64_t S[3], O[3];
    int k[3], s[3], p[3], d[3];
    const int64_t *idx;
    double *out;
} prob_t;

static int fill_prob(prob_t *P, const double *x, const double *w, const double *b,
                     int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1,
                     int k2, const int stride[3], const int pad[3], const int dil[3],
                     const int out_pad[3], int groups, int transposed) {
    memset(P, 0, sizeof(*P));
    if (!x || !w || !stride || !pad || !dil) return -1;
    if (N <= 0 || Cin <= 0 || Cout <= 0 || groups <= 0) return -1;
    if (Cin % groups || Cout % groups) return -1;
    P->x = x;
    P->w = w;
    P->b = b;
    P->N = N;
    P->Cin = Cin;
    P->Cout = Cout;
    P->G = groups;
    P->S[0] = S0;
    P->S[1] = S1;
    P->S[2] = S2;
    P->k[0] = k0;
    P->k[1] = k1;
    P->k[2] = k2;
    for (int a = 0; a < 3; ++a) {
        P->s[a] = stride[a];
        P->p[a] = pad[a];
        P->d[a] = dil[a];
        int op = transposed ? (out_pad ? out_pad[a] : 0) : 0;
        P->O[a] = transposed ? oracle_convT_out_len(P->S[a], P->k[a], P->s[a], P->p[a], P->d[a], op)
                             : oracle_conv_out_len(P->S[a], P->k[a], P->s[a], P->p[a], P->d[a]);
        if (P->O[a] <= 0) return -1;
    }
    return 0;
}

/* conv3d at one output point: bias + sum over the group's input channels and
 * all taps whose input index lies inside the input (zero padding outside). */
static double conv_point(const prob_t *P, int n, int oc, int64_t o0, int64_t o1, int64_t o2) {
    const int cin_g = P->Cin / P->G, cout_g = P->Cout / P->G;
    const int grp = oc / cout_g;
    const int64_t S0 = P->S[0], S1 = P->S[1], S2 = P->S[2];
    const int K0 = P->k[0], K1 = P->k[1], K2 = P->k[2];
    double acc = P->b ? P->b[oc] : 0.0;
    for (int icl = 0; icl < cin_g; ++icl) {
        const int ic = grp * cin_g + icl;
        const double *xc = P->x + ((int64_t)n * P->Cin + ic) * S0 * S1 * S2;
        const double *wc = P->w + ((int64_t)oc * cin_g + icl) * K0 * K1 * K2;
        for (int a = 0; a < K0; ++a) {
            const int64_t i0 = o0 * P->s[0] - P->p[0] + (int64_t)P->d[0] * a;
            if (i0 < 0 || i0 >= S0) continue;
            for (int b = 0; b < K1; ++b) {
                const int64_t i1 = o1 * P->s[1] - P->p[1] + (int64_t)P->d[1] * b;
                if (i1 < 0 || i1 >= S1) continue;
                for (int c = 0; c < K2; ++c) {
                    const int64_t i2 = o2 * P->s[2] - P->p[2] + (int64_t)P->d[2] * c;
                    if (i2 < 0 || i2 >= S2) continue;
                    acc += wc[((int64_t)a * K1 + b) * K2 + c] * xc[(i0 * S1 + i1) * S2 + i2];
                }
            }
        }
    }
    return acc;
}

/* transposed conv at one output point, receive form: tap k of axis a
 * contributes iff (z + p - d k) is divisible by s and the quotient is a valid
 * input index. */
static double convT_point(const prob_t *P, int n, int oc, int64_t z0, int64_t z1, int64_t z2) {
    const int cin_g = P->Cin / P->G, cout_g = P->Cout / P->G;
    const int grp = oc / cout_g, ocl = oc % cout_g;
    const int64_t S0 = P->S[0], S1 = P->S[1], S2 = P->S[2];
    const int K0 = P->k[0], K1 = P->k[1], K2 = P->k[2];
    double acc = P->b ? P->b[oc] : 0.0;
    for (int icl = 0; icl < cin_g; ++icl) {
        const int ic = grp * cin_g + icl;
        const double *xc = P->x + ((int64_t)n * P->Cin + ic) * S0 * S1 * S2;
        const double *wc = P->w + ((int64_t)ic * cout_g + ocl) * K0 * K1 * K2;
        for (int a = 0; a < K0; ++a) {
            const int64_t t0 = z0 + P->p[0] - (int64_t)P->d[0] * a;
            if (t0 % P->s[0] != 0) continue;
            const int64_t i0 = t0 / P->s[0];
            if (i0 < 0 || i0 >= S0) continue;
            for (int b = 0; b < K1; ++b) {
                const int64_t t1 = z1 + P->p[1] - (int64_t)P->d[1] * b;
                if (t1 % P->s[1] != 0) continue;
                const int64_t i1 = t1 / P->s[1];
                if (i1 < 0 || i1 >= S1) continue;
                for (int c = 0; c < K2; ++c) {
                    const int64_t t2 = z2 + P->p[2] - (int64_t)P->d[2] * c;
                    if (t2 % P->s[2] != 0) continue;
                    const int64_t i2 = t2 / P->s[2];
                    if (i2 < 0 || i2 >= S2) continue;
                    acc += wc[((int64_t)a * K1 + b) * K2 + c] * xc[(i0 * S1 + i1) * S2 + i2];
                }
            }
        }
    }
    return acc;
}

typedef double (*point_fn)(const prob_t *, int, int, int64_t, int64_t, int64_t);

typedef struct {
    const prob_t *P;
    point_fn f;
} full_ctx;

/* one work item = one (n, oc) slice of the output */
static void full_range(void *vctx, int64_t begin, int64_t end) {
    const full_ctx *c = (const full_ctx *)vctx;
    const prob_t *P = c->P;
    const int64_t O0 = P->O[0], O1 = P->O[1], O2 = P->O[2];
    for (int64_t it = begin; it < end; ++it) {
        const int n = (int)(it / P->Cout), oc = (int)(it % P->Cout);
        double *ys = P->y + it * O0 * O1 * O2;
        for (int64_t o0 = 0; o0 < O0; ++o0)
            for (int64_t o1 = 0; o1 < O1; ++o1)
                for (int64_t o2 = 0; o2 < O2; ++o2)
                    ys[(o0 * O1 + o1) * O2 + o2] = c->f(P, n, oc, o0, o1, o2);
    }
}

static void at_range(void *vctx, int64_t begin, int64_t end) {
    const full_ctx *c = (const full_ctx *)vctx;
    const prob_t *P = c->P;
    const int64_t O0 = P->O[0], O1 = P->O[1], O2 = P->O[2];
    for (int64_t i = begin; i < end; ++i) {
        int64_t f = P->idx[i];
        const int64_t o2 = f % O2;
        f /= O2;
        const int64_t o1 = f % O1;
        f /= O1;
        const int64_t o0 = f % O0;
        f /= O0;
        const int oc = (int)(f % P->Cout);
        const int n = (int)(f / P->Cout);
        P->out[i] = c->f(P, n, oc, o0, o1, o2);
    }
}

static int check_idx(const int64_t *idx, int64_t count, int64_t total) {
    if (count < 0 || (count > 0 && !idx)) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (idx[i] < 0 || idx[i] >= total) return -1;
    return 0;
}

int oracle_conv3d(const double *x, const double *w, const double *b, double *y, int N, int Cin,
                  int S0, int S1, int S2, int Cout, int k0, int k1, int k2, const int stride[3],
                  const int pad[3], const int dil[3], int groups, int nthreads) {
    prob_t P;
    if (!y || fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, NULL,
                        groups, 0))
        return -1;
    P.y = y;
    full_ctx c = {&P, conv_point};
    par_for((int64_t)N * Cout, nthreads, 1, full_range, &c);
    return 0;
}

int oracle_conv3d_at(const double *x, const double *w, const double *b, int N, int Cin, int S0,
                     int S1, int S2, int Cout, int k0, int k1, int k2, const int stride[3],
                     const int pad[3], const int dil[3], int groups, const int64_t *idx,
                     int64_t count, double *out, int nthreads) {
    prob_t P;
    if (fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, NULL, groups,
                  0))
        return -1;
    if (check_idx(idx, count, (int64_t)N * Cout * P.O[0] * P.O[1] * P.O[2]) || (count && !out))
        return -1;
    P.idx = idx;
    P.out = out;
    full_ctx c = {&P, conv_point};
    par_for(count, nthreads, 16, at_range, &c);
    return 0;
}

int oracle_conv_transpose3d(const double *x, const double *w, const double *b, double *y, int N,
                            int Cin, int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                            const int stride[3], const int pad[3], const int dil[3],
                            const int out_pad[3], int groups, int nthreads) {
    prob_t P;
    if (!y || fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil,
                        out_pad, groups, 1))
        return -1;
    P.y = y;
    full_ctx c = {&P, convT_point};
    par_for((int64_t)N * Cout, nthreads, 1, full_range, &c);
    return 0;
}

int oracle_conv_transpose3d_at(const double *x, const double *w, const double *b, int N, int Cin,
                               int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                               const int stride[3], const int pad[3], const int dil[3],
                               const int out_pad[3], int groups, const int64_t *idx,
                               int64_t count, double *out, int nthreads) {
    prob_t P;
    if (fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, out_pad,
                  groups, 1))
        return -1;
    if (check_idx(idx, count, (int64_t)N * Cout * P.O[0] * P.O[1] * P.O[2]) || (count && !out))
        return -1;
    P.idx = idx;
    P.out = out;
    full_ctx c = {&P, convT_point};
    par_for(count, nthreads, 16, at_range, &c);
    return 0;
}

int oracle_conv_transpose3d_scatter(const double *x, const double *w, const double *b, double *y,
                                    int N, int Cin, int S0, int S1, int S2, int Cout, int k0,
                                    int k1, int k2, const int stride[3], const int pad[3],
                                    const int dil[3], const int out_pad[3], int groups) {
    prob_t P;
    if (!y || fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil,
                        out_pad, groups, 1))
        return -1;
    const int cin_g = Cin / groups, cout_g = Cout / groups;
    const int64_t O0 = P.O[0], O1 = P.O[1], O2 = P.O[2];
    const int64_t ovol = O0 * O1 * O2;
    memset(y, 0, sizeof(double) * (size_t)((int64_t)N * Cout * ovol));
    for (int n = 0; n < N; ++n)
        for (int ic = 0; ic < Cin; ++ic) {
            const int grp = ic / cin_g;
            const double *xc = x + ((int64_t)n * Cin + ic) * S0 * S1 * S2;
            for (int64_t i0 = 0; i0 < S0; ++i0)
                for (int64_t i1 = 0; i1 < S1; ++i1)
                    for (int64_t i2 = 0; i2 < S2; ++i2) {
                        const double xv = xc[(i0 * S1 + i1) * S2 + i2];
                        for (int ocl = 0; ocl < cout_g; ++ocl) {
                            const int oc = grp * cout_g + ocl;
                            double *yc = y + ((int64_t)n * Cout + oc) * ovol;
                            const double *wc = w + ((int64_t)ic * cout_g + ocl) * k0 * k1 * k2;
                            for (int a = 0; a < k0; ++a) {
                                const int64_t z0 = i0 * stride[0] - pad[0] + (int64_t)dil[0] * a;
                                if (z0 < 0 || z0 >= O0) continue;
                                for (int bb = 0; bb < k1; ++bb) {
                                    const int64_t z1 =
                                        i1 * stride[1] - pad[1] + (int64_t)dil[1] * bb;
                                    if (z1 < 0 || z1 >= O1) continue;
                                    for (int c = 0; c < k2; ++c) {
                                        const int64_t z2 =
                                            i2 * stride[2] - pad[2] + (int64_t)dil[2] * c;
                                        if (z2 < 0 || z2 >= O2) continue;
                                        yc[(z0 * O1 + z1) * O2 + z2] +=
                                            wc[((int64_t)a * k1 + bb) * k2 + c] * xv;
                                    }
                                }
                            }
                        }
                    }
        }
    if (b)
        for (int n = 0; n < N; ++n)
            for (int oc = 0; oc < Cout; ++oc) {
                double *yc = y + ((int64_t)n * Cout + oc) * ovol;
                for (int64_t i = 0; i < ovol; ++i) yc[i] += b[oc];
            }
    return 0;
}

/* ------------------------------------------------------------------ */
/* pooling, logsumexp, relu, batchnorm                                  */
/* ------------------------------------------------------------------ */
static int pool2(const double *t, double *out, int N, int C, int L0, int L1, int L2, int is_max) {
    if (!t || !out || N <= 0 || C <= 0) return -1;
    const int64_t P0 = L0 / 2, P1 = L1 / 2, P2 = L2 / 2;
    if (P0 <= 0 || P1 <= 0 || P2 <= 0) return -1;
    for (int64_t nc = 0; nc < (int64_t)N * C; ++nc) {
        const double *tc = t + nc * (int64_t)L0 * L1 * L2;
        double *oc = out + nc * P0 * P1 * P2;
        for (int64_t q0 = 0; q0 < P0; ++q0)
            for (int64_t q1 = 0; q1 < P1; ++q1)
                for (int64_t q2 = 0; q2 < P2; ++q2) {
                    double acc = is_max ? -INFINITY : 0.0;
                    for (int a = 0; a < 2; ++a)
                        for (int b = 0; b < 2; ++b)
                            for (int c = 0; c < 2; ++c) {
                                const double v =
                                    tc[((2 * q0 + a) * L1 + (2 * q1 + b)) * (int64_t)L2 + 2 * q2 + c];
                                if (is_max)
                                    acc = v > acc ? v : acc;
                                else
                                    acc += v;
                            }
                    oc[(q0 * P1 + q1) * P2 + q2] = is_max ? acc : acc / 8.0;
                }
    }
    return 0;
}

int oracle_maxpool3d_2(const double *t, double *out, int N, int C, int L0, int L1, int L2) {
    return pool2(t, out, N, C, L0, L1, L2, 1);
}

int oracle_avgpool3d_2(const double *t, double *out, int N, int C, int L0, int L1, int L2) {
    return pool2(t, out, N, C, L0, L1, L2, 0);
}

int oracle_logsumexp_channels(const double *t, double *out, int N, int C, int64_t L) {
    if (!t || !out || N <= 0 || C <= 0 || L <= 0) return -1;
    for (int n = 0; n < N; ++n)
        for (int64_t s = 0; s < L; ++s) {
            const double *tn = t + (int64_t)n * C * L + s;
            double m = tn[0];
            for (int c = 1; c < C; ++c) m = tn[(int64_t)c * L] > m ? tn[(int64_t)c * L] : m;
            double acc = 0.0;
            for (int c = 0; c < C; ++c) acc += exp(tn[(int64_t)c * L] - m);
            out[(int64_t)n * L + s] = m + log(acc);
        }
    return 0;
}

void oracle_relu(double *t, int64_t n) {
    for (int64_t i = 0; i < n; ++i) t[i] = t[i] > 0.0 ? t[i] : 0.0;
}

int oracle_batchnorm3d_train(const double *t, double *out, int N, int C, int64_t L,
                             const double *gamma, const double *beta, double eps,
                             double *mean_out, double *var_out) {
    if (!t || !out || N <= 0 || C <= 0 || L <= 0 || !(eps >= 0.0)) return -1;
    const double cnt = (double)N * (double)L;
    for (int c = 0; c < C; ++c) {
        double sum = 0.0;
        for (int n = 0; n < N; ++n) {
            const double *tc = t + ((int64_t)n * C + c) * L;
            for (int64_t i = 0; i < L; ++i) sum += tc[i];
        }
        const double mean = sum / cnt;
        double ss = 0.0;
        for (int n = 0; n < N; ++n) {
            const double *tc = t + ((int64_t)n * C + c) * L;
            for (int64_t i = 0; i < L; ++i) ss += (tc[i] - mean) * (tc[i] - mean);
        }
        const double var = ss / cnt; /* biased: divide by the element count */
        const double g = gamma ? gamma[c] : 1.0, be = beta ? beta[c] : 0.0;
        const double inv = 1.0 / sqrt(var + eps);
        for (int n = 0; n < N; ++n) {
            const double *tc = t + ((int64_t)n * C + c) * L;
            double *oc = out + ((int64_t)n * C + c) * L;
            for (int64_t i = 0; i < L; ++i) oc[i] = (tc[i] - mean) * inv * g + be;
        }
        if (mean_out) mean_out[c] = mean;
        if (var_out) var_out[c] = var;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* composites                                                           */
/* ------------------------------------------------------------------ */
int oracle_convT_bn_avgpool(const double *x, const double *w, const double *b, const double *gamma,
                            const double *beta, double eps, double *y, int N, int Cin, int S0,
                            int S1, int S2, int Cout, int k0, int k1, int k2, const int stride[3],
                            const int pad[3], const int dil[3], const int out_pad[3], int groups,
                            int nthreads) {
    prob_t P;
    if (!y || fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil,
                        out_pad, groups, 1))
        return -1;
    const int64_t O0 = P.O[0], O1 = P.O[1], O2 = P.O[2];
    const int64_t Q0 = O0 / 2, Q1 = O1 / 2, Q2 = O2 / 2;
    if (Q0 / 2 <= 0 || Q1 / 2 <= 0 || Q2 / 2 <= 0) return -1;
    const int64_t nc = (int64_t)N * Cout;
    double *t = (double *)malloc(sizeof(double) * (size_t)(nc * O0 * O1 * O2));
    double *u = (double *)malloc(sizeof(double) * (size_t)(nc * O0 * O1 * O2));
    if (!t || !u) {
        free(t);
        free(u);
        return -1;
    }
    int rc = oracle_conv_transpose3d(x, w, b, t, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad,
                                     dil, out_pad, groups, nthreads);
    if (!rc) rc = oracle_batchnorm3d_train(t, u, N, Cout, O0 * O1 * O2, gamma, beta, eps, NULL, NULL);
    if (!rc) rc = oracle_avgpool3d_2(u, t, N, Cout, (int)O0, (int)O1, (int)O2);
    if (!rc) rc = oracle_avgpool3d_2(t, y, N, Cout, (int)Q0, (int)Q1, (int)Q2);
    free(t);
    free(u);
    return rc;
}

int oracle_batchnorm3d_eval(const double *t, double *out, int N, int C, int64_t L,
                            const double *rmean, const double *rvar, const double *gamma,
                            const double *beta, double eps) {
    if (!t || !out || !rmean || !rvar || N <= 0 || C <= 0 || L <= 0 || !(eps >= 0.0)) return -1;
    for (int c = 0; c < C; ++c) {
        const double g = gamma ? gamma[c] : 1.0, be = beta ? beta[c] : 0.0;
        const double inv = 1.0 / sqrt(rvar[c] + eps);
        for (int n = 0; n < N; ++n) {
            const double *tc = t + ((int64_t)n * C + c) * L;
            double *oc = out + ((int64_t)n * C + c) * L;
            for (int64_t i = 0; i < L; ++i) oc[i] = (tc[i] - rmean[c]) * inv * g + be;
        }
    }
    return 0;
}

int oracle_convT_bneval_avgpool(const double *x, const double *w, const double *b,
                                const double *rmean, const double *rvar, const double *gamma,
                                const double *beta, double eps, double *y, int N, int Cin,
                                int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                                const int stride[3], const int pad[3], const int dil[3],
                                const int out_pad[3], int groups, int nthreads) {
    prob_t P;
    if (!y || fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil,
                        out_pad, groups, 1))
        return -1;
    const int64_t O0 = P.O[0], O1 = P.O[1], O2 = P.O[2];
    const int64_t Q0 = O0 / 2, Q1 = O1 / 2, Q2 = O2 / 2;
    if (Q0 / 2 <= 0 || Q1 / 2 <= 0 || Q2 / 2 <= 0) return -1;
    const int64_t nc = (int64_t)N * Cout;
    double *t = (double *)malloc(sizeof(double) * (size_t)(nc * O0 * O1 * O2));
    double *u = (double *)malloc(sizeof(double) * (size_t)(nc * O0 * O1 * O2));
    if (!t || !u) {
        free(t);
        free(u);
        return -1;
    }
    int rc = oracle_conv_transpose3d(x, w, b, t, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad,
                                     dil, out_pad, groups, nthreads);
    if (!rc)
        rc = oracle_batchnorm3d_eval(t, u, N, Cout, O0 * O1 * O2, rmean, rvar, gamma, beta, eps);
    if (!rc) rc = oracle_avgpool3d_2(u, t, N, Cout, (int)O0, (int)O1, (int)O2);
    if (!rc) rc = oracle_avgpool3d_2(t, y, N, Cout, (int)Q0, (int)Q1, (int)Q2);
    free(t);
    free(u);
    return rc;
}

/* per-(n, c) slice statistics for the sampled BN composite */
typedef struct {
    const prob_t *P;
    double *mean, *m2; /* [N*Cout] */
    int64_t slice;
} stat_ctx;

static void stat_range(void *vctx, int64_t begin, int64_t end) {
    const stat_ctx *c = (const stat_ctx *)vctx;
    const prob_t *P = c->P;
    const int64_t O0 = P->O[0], O1 = P->O[1], O2 = P->O[2];
    double *buf = (double *)malloc(sizeof(double) * (size_t)c->slice);
    if (!buf) return;
    for (int64_t it = begin; it < end; ++it) {
        const int n = (int)(it / P->Cout), oc = (int)(it % P->Cout);
        for (int64_t o0 = 0; o0 < O0; ++o0)
            for (int64_t o1 = 0; o1 < O1; ++o1)
                for (int64_t o2 = 0; o2 < O2; ++o2)
                    buf[(o0 * O1 + o1) * O2 + o2] = convT_point(P, n, oc, o0, o1, o2);
        double s = 0.0;
        for (int64_t i = 0; i < c->slice; ++i) s += buf[i];
        const double m = s / (double)c->slice;
        double ss = 0.0;
        for (int64_t i = 0; i < c->slice; ++i) ss += (buf[i] - m) * (buf[i] - m);
        c->mean[it] = m;
        c->m2[it] = ss;
    }
    free(buf);
}

typedef struct {
    const prob_t *P;
    const double *mean, *var, *gamma, *beta;
    double eps;
} bnpool_ctx;

/* value of BN(convT) at one full-resolution position */
static double bn_value(const bnpool_ctx *c, int n, int oc, int64_t z0, int64_t z1, int64_t z2) {
    const double v = convT_point(c->P, n, oc, z0, z1, z2);
    const double g = c->gamma ? c->gamma[oc] : 1.0, be = c->beta ? c->beta[oc] : 0.0;
    return (v - c->mean[oc]) * (1.0 / sqrt(c->var[oc] + c->eps)) * g + be;
}

static void bnpool_range(void *vctx, int64_t begin, int64_t end) {
    const bnpool_ctx *c = (const bnpool_ctx *)vctx;
    const prob_t *P = c->P;
    const int64_t R0 = P->O[0] / 2 / 2, R1 = P->O[1] / 2 / 2, R2 = P->O[2] / 2 / 2;
    for (int64_t i = begin; i < end; ++i) {
        int64_t f = P->idx[i];
        const int64_t q2 = f % R2;
        f /= R2;
        const int64_t q1 = f % R1;
        f /= R1;
        const int64_t q0 = f % R0;
        f /= R0;
        const int oc = (int)(f % P->Cout);
        const int n = (int)(f / P->Cout);
        /* second AvgPool3d(2) over first-level outputs 2q+e, each of which is
         * the first AvgPool3d(2) over positions 2(2q+e)+f' */
        double outer = 0.0;
        for (int e0 = 0; e0 < 2; ++e0)
            for (int e1 = 0; e1 < 2; ++e1)
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int64_t r0 = 2 * q0 + e0, r1 = 2 * q1 + e1, r2 = 2 * q2 + e2;
                    double inner = 0.0;
                    for (int f0 = 0; f0 < 2; ++f0)
                        for (int f1 = 0; f1 < 2; ++f1)
                            for (int f2 = 0; f2 < 2; ++f2)
                                inner += bn_value(c, n, oc, 2 * r0 + f0, 2 * r1 + f1, 2 * r2 + f2);
                    outer += inner / 8.0;
                }
        P->out[i] = outer / 8.0;
    }
}

int oracle_convT_bn_avgpool_at(const double *x, const double *w, const double *b,
                               const double *gamma, const double *beta, double eps, int N, int Cin,
                               int S0, int S1, int S2, int Cout, int k0, int k1, int k2,
                               const int stride[3], const int pad[3], const int dil[3],
                               const int out_pad[3], int groups, const int64_t *idx, int64_t count,
                               double *out, double *mean_out, double *var_out, int nthreads) {
    prob_t P;
    if (fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, out_pad,
                  groups, 1) ||
        !(eps >= 0.0))
        return -1;
    const int64_t R0 = P.O[0] / 2 / 2, R1 = P.O[1] / 2 / 2, R2 = P.O[2] / 2 / 2;
    if (R0 <= 0 || R1 <= 0 || R2 <= 0) return -1;
    if (check_idx(idx, count, (int64_t)N * Cout * R0 * R1 * R2) || (count && !out)) return -1;
    const int64_t nc = (int64_t)N * Cout;
    const int64_t slice = P.O[0] * P.O[1] * P.O[2];
    double *sm = (double *)malloc(sizeof(double) * (size_t)nc);
    double *s2 = (double *)malloc(sizeof(double) * (size_t)nc);
    double *mean = (double *)malloc(sizeof(double) * (size_t)Cout);
    double *var = (double *)malloc(sizeof(double) * (size_t)Cout);
    if (!sm || !s2 || !mean || !var) {
        free(sm);
        free(s2);
        free(mean);
        free(var);
        return -1;
    }
    stat_ctx sc = {&P, sm, s2, slice};
    par_for(nc, nthreads, 1, stat_range, &sc);
    /* combine the N slices of each channel exactly (pairwise mean/M2 update),
     * in the fixed order n = 0 .. N-1 */
    for (int oc = 0; oc < Cout; ++oc) {
        double cnt = (double)slice, m = sm[oc], M2 = s2[oc];
        for (int n = 1; n < N; ++n) {
            const double nb = (double)slice, mb = sm[(int64_t)n * Cout + oc];
            const double M2b = s2[(int64_t)n * Cout + oc];
            const double tot = cnt + nb, delta = mb - m;
            m += delta * nb / tot;
            M2 += M2b + delta * delta * cnt * nb / tot;
            cnt = tot;
        }
        mean[oc] = m;
        var[oc] = M2 / cnt;
        if (mean_out) mean_out[oc] = mean[oc];
        if (var_out) var_out[oc] = var[oc];
    }
    P.idx = idx;
    P.out = out;
    bnpool_ctx bc = {&P, mean, var, gamma, beta, eps};
    par_for(count, nthreads, 4, bnpool_range, &bc);
    free(sm);
    free(s2);
    free(mean);
    free(var);
    return 0;
}

int oracle_convT_bneval_avgpool_at(const double *x, const double *w, const double *b,
                                   const double *rmean, const double *rvar, const double *gamma,
                                   const double *beta, double eps, int N, int Cin, int S0, int S1,
                                   int S2, int Cout, int k0, int k1, int k2, const int stride[3],
                                   const int pad[3], const int dil[3], const int out_pad[3],
                                   int groups, const int64_t *idx, int64_t count, double *out,
                                   int nthreads) {
    prob_t P;
    if (!rmean || !rvar ||
        fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, out_pad,
                  groups, 1) ||
        !(eps >= 0.0))
        return -1;
    const int64_t R0 = P.O[0] / 2 / 2, R1 = P.O[1] / 2 / 2, R2 = P.O[2] / 2 / 2;
    if (R0 <= 0 || R1 <= 0 || R2 <= 0) return -1;
    if (check_idx(idx, count, (int64_t)N * Cout * R0 * R1 * R2) || (count && !out)) return -1;
    P.idx = idx;
    P.out = out;
    /* the literal two-stage pooling of BN(convT) at every sampled output, with
     * the running statistics in place of batch statistics */
    bnpool_ctx bc = {&P, rmean, rvar, gamma, beta, eps};
    par_for(count, nthreads, 4, bnpool_range, &bc);
    return 0;
}

int oracle_conv_maxpool_lse_relu(const double *x, const double *w, const double *b, double *y,
                                 int N, int Cin, int S0, int S1, int S2, int Cout, int k0, int k1,
                                 int k2, const int stride[3], const int pad[3], const int dil[3],
                                 int groups, int nthreads) {
    prob_t P;
    if (!y || fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, NULL,
                        groups, 0))
        return -1;
    const int64_t O0 = P.O[0], O1 = P.O[1], O2 = P.O[2];
    const int64_t Q0 = O0 / 2, Q1 = O1 / 2, Q2 = O2 / 2;
    if (Q0 <= 0 || Q1 <= 0 || Q2 <= 0) return -1;
    double *t = (double *)malloc(sizeof(double) * (size_t)((int64_t)N * Cout * O0 * O1 * O2));
    double *u = (double *)malloc(sizeof(double) * (size_t)((int64_t)N * Cout * Q0 * Q1 * Q2));
    if (!t || !u) {
        free(t);
        free(u);
        return -1;
    }
    int rc = oracle_conv3d(x, w, b, t, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil,
                           groups, nthreads);
    if (!rc) rc = oracle_maxpool3d_2(t, u, N, Cout, (int)O0, (int)O1, (int)O2);
    if (!rc) rc = oracle_logsumexp_channels(u, y, N, Cout, Q0 * Q1 * Q2);
    if (!rc) oracle_relu(y, (int64_t)N * Q0 * Q1 * Q2);
    free(t);
    free(u);
    return rc;
}

typedef struct {
    const prob_t *P;
    double *scratch; /* per sample: Cout pooled values, allocated per range */
} mlr_ctx;

static void mlr_range(void *vctx, int64_t begin, int64_t end) {
    const mlr_ctx *c = (const mlr_ctx *)vctx;
    const prob_t *P = c->P;
    const int64_t Q0 = P->O[0] / 2, Q1 = P->O[1] / 2, Q2 = P->O[2] / 2;
    double *v = (double *)malloc(sizeof(double) * (size_t)P->Cout);
    if (!v) return;
    for (int64_t i = begin; i < end; ++i) {
        int64_t f = P->idx[i];
        const int64_t q2 = f % Q2;
        f /= Q2;
        const int64_t q1 = f % Q1;
        f /= Q1;
        const int64_t q0 = f % Q0;
        const int n = (int)(f / Q0);
        /* MaxPool3d(2,2) of each channel at pooled position q */
        for (int oc = 0; oc < P->Cout; ++oc) {
            double m = -INFINITY;
            for (int a = 0; a < 2; ++a)
                for (int b = 0; b < 2; ++b)
                    for (int e = 0; e < 2; ++e) {
                        const double t = conv_point(P, n, oc, 2 * q0 + a, 2 * q1 + b, 2 * q2 + e);
                        m = t > m ? t : m;
                    }
            v[oc] = m;
        }
        /* logsumexp over channels, then ReLU */
        double m = v[0];
        for (int oc = 1; oc < P->Cout; ++oc) m = v[oc] > m ? v[oc] : m;
        double acc = 0.0;
        for (int oc = 0; oc < P->Cout; ++oc) acc += exp(v[oc] - m);
        const double l = m + log(acc);
        P->out[i] = l > 0.0 ? l : 0.0;
    }
    free(v);
}

int oracle_conv_maxpool_lse_relu_at(const double *x, const double *w, const double *b, int N,
                                    int Cin, int S0, int S1, int S2, int Cout, int k0, int k1,
                                    int k2, const int stride[3], const int pad[3],
                                    const int dil[3], int groups, const int64_t *idx,
                                    int64_t count, double *out, int nthreads) {
    prob_t P;
    if (fill_prob(&P, x, w, b, N, Cin, S0, S1, S2, Cout, k0, k1, k2, stride, pad, dil, NULL, groups,
                  0))
        return -1;
    const int64_t Q0 = P.O[0] / 2, Q1 = P.O[1] / 2, Q2 = P.O[2] / 2;
    if (Q0 <= 0 || Q1 <= 0 || Q2 <= 0) return -1;
    if (check_idx(idx, count, (int64_t)N * Q0 * Q1 * Q2) || (count && !out)) return -1;
    P.idx = idx;
    P.out = out;
    mlr_ctx c = {&P, NULL};
    par_for(count, nthreads, 4, mlr_range, &c);
    return 0;
}
