/*
 * ct_oracle_mt.c -- TEST AND BENCHMARK INFRASTRUCTURE ONLY.
 *
 * The CPU baseline on all host cores: the scatter definition of the forward
 * transposed convolution that ct_oracle.c evaluates, with its work split over
 * POSIX threads by output slice (n, oc).  Each thread owns whole slices
 * y[n, oc, :], so no two threads write the same output and no atomics are
 * needed.  For its slice a thread runs the scatter rule of the pages
 * ([l1_p79] out[i*s - p + k*d] += in[i]*w[k]; [l1_p72] the grouped channel
 * mapping, no kernel flip) over the input channels of the slice's group, then
 * adds the bias.  Arithmetic in double, as the parity oracle.
 *
 * It exists to time the oracle with every host core busy (the benchmark's
 * CPU baseline), not to check results: the parity tests use ct_oracle.c.  A
 * test compares the two on small shapes.  Nothing in the product path links,
 * loads or calls this file, and it shares no code with the CUDA library or
 * with ct_oracle.c.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    int64_t N, C_in, C_out, G;
    int64_t Li[3], Lo[3], K[3], S[3], P[3], D[3];
    const double *x, *w, *bias;
    double *y;
    int64_t first, last;        /* output slices t = n * C_out + oc in [first, last) */
} mt_job;

/* [l1_p79] output-length formula, per dimension */
static int64_t mt_out_len(int64_t L_in, int64_t k, int64_t s, int64_t p, int64_t op, int64_t dl)
{
    return (L_in - 1) * s - 2 * p + dl * (k - 1) + op + 1;
}

static void *mt_worker(void *arg)
{
    const mt_job *j = (const mt_job *)arg;
    const int64_t Cig = j->C_in / j->G, Cog = j->C_out / j->G;
    const int64_t in_sp = j->Li[0] * j->Li[1] * j->Li[2];
    const int64_t out_sp = j->Lo[0] * j->Lo[1] * j->Lo[2];
    const int64_t kvol = j->K[0] * j->K[1] * j->K[2];
    for (int64_t t = j->first; t < j->last; ++t) {
        const int64_t n = t / j->C_out, oc = t % j->C_out;
        const int64_t g = oc / Cog, ocl = oc % Cog;
        double *yo = j->y + t * out_sp;
        for (int64_t e = 0; e < out_sp; ++e) yo[e] = 0.0;
        for (int64_t ic = g * Cig; ic < (g + 1) * Cig; ++ic) {
            const double *xc = j->x + (n * j->C_in + ic) * in_sp;
            const double *wk = j->w + (ic * Cog + ocl) * kvol;
            for (int64_t i0 = 0; i0 < j->Li[0]; ++i0)
            for (int64_t i1 = 0; i1 < j->Li[1]; ++i1)
            for (int64_t i2 = 0; i2 < j->Li[2]; ++i2) {
                const double xv = xc[(i0 * j->Li[1] + i1) * j->Li[2] + i2];
                for (int64_t k0 = 0; k0 < j->K[0]; ++k0) {
                    const int64_t o0 = i0 * j->S[0] - j->P[0] + k0 * j->D[0];
                    if (o0 < 0 || o0 >= j->Lo[0]) continue;
                    for (int64_t k1 = 0; k1 < j->K[1]; ++k1) {
                        const int64_t o1 = i1 * j->S[1] - j->P[1] + k1 * j->D[1];
                        if (o1 < 0 || o1 >= j->Lo[1]) continue;
                        for (int64_t k2 = 0; k2 < j->K[2]; ++k2) {
                            const int64_t o2 = i2 * j->S[2] - j->P[2] + k2 * j->D[2];
                            if (o2 < 0 || o2 >= j->Lo[2]) continue;
                            yo[(o0 * j->Lo[1] + o1) * j->Lo[2] + o2] += xv * wk[(k0 * j->K[1] + k1) * j->K[2] + k2];
                        }
                    }
                }
            }
        }
        if (j->bias)
            for (int64_t e = 0; e < out_sp; ++e) yo[e] += j->bias[oc];
    }
    return NULL;
}

/* Same arguments and layouts as ora_conv_transpose in ct_oracle.c, plus the
 * number of threads (>= 1).  Returns 0, 1 on invalid arguments, 3 if a
 * thread could not be started. */
int ora_mt_conv_transpose(int nthreads, int nd, int64_t N, int64_t C_in, int64_t C_out, int64_t G,
                          const int64_t *L_in, const int64_t *K, const int64_t *S, const int64_t *P,
                          const int64_t *OP, const int64_t *DL, const double *x, const double *w,
                          const double *bias, double *y)
{
    if (nthreads < 1 || nd < 1 || nd > 3) return 1;
    if (N < 0 || C_in <= 0 || C_out <= 0 || G <= 0 || C_in % G || C_out % G) return 1;
    mt_job base;
    base.N = N; base.C_in = C_in; base.C_out = C_out; base.G = G;
    for (int d = 0; d < 3; ++d) {
        base.Li[d] = 1; base.Lo[d] = 1; base.K[d] = 1; base.S[d] = 1; base.P[d] = 0; base.D[d] = 1;
    }
    for (int d = 0; d < nd; ++d) {
        const int e = 3 - nd + d;
        if (L_in[d] <= 0 || K[d] <= 0 || S[d] <= 0 || DL[d] <= 0 || P[d] < 0 || OP[d] < 0) return 1;
        base.Li[e] = L_in[d]; base.K[e] = K[d]; base.S[e] = S[d]; base.P[e] = P[d]; base.D[e] = DL[d];
        base.Lo[e] = mt_out_len(L_in[d], K[d], S[d], P[d], OP[d], DL[d]);
        if (base.Lo[e] <= 0) return 1;
    }
    base.x = x; base.w = w; base.bias = bias; base.y = y;
    const int64_t slices = N * C_out;
    if (slices == 0) return 0;
    if ((int64_t)nthreads > slices) nthreads = (int)slices;
    mt_job *jobs = (mt_job *)malloc(sizeof(mt_job) * (size_t)nthreads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return 3;
    }
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = base;
        jobs[i].first = slices * i / nthreads;
        jobs[i].last = slices * (i + 1) / nthreads;
    }
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, mt_worker, &jobs[i]) != 0) {
            rc = 3;
            break;
        }
        ++started;
    }
    mt_worker(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    if (rc == 3)   /* finish the slices of the threads that did not start */
        for (int i = started + 1; i < nthreads; ++i) mt_worker(&jobs[i]);
    free(jobs);
    free(th);
    return 0;
}
