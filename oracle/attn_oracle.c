/*
 * Oracle: fp64 tree/DAG-packed attention, forward and backward, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously correct code used to check the CUDA
 * path; the library never links or calls it.  It shares no code, header or table with the
 * CUDA path or its planner.
 *
 * What it computes (Octopus, arXiv 2611.06956, Section 3.3 Eq. 4 and Section 3.4; HARTS,
 * arXiv 2608.28158, Section 3.4 and Section 4.2 Eq. 21-22): for each listed query row r and
 * query head h, with KV head g = h / (Hq / Hkv) and vis(r) the row's visible set given as
 * disjoint [lo, hi) row intervals,
 *
 *   s_j   = scale * <Q[r,h], K[j,g]>                      j in vis(r)
 *   lse   = ln sum_j exp(s_j)
 *   p_j   = exp(s_j - lse)
 *   O     = sum_j p_j V[j,g]
 *
 * and, for a given upstream gradient dO (the exact adjoint of the above; gradients through
 * a shared or mounted row are summed over every reader: Octopus Section 3.4 "differentiable
 * mount edges", HARTS Section 3.4 gather backward):
 *
 *   delta   = <dO[r,h], O[r,h]>
 *   dS_j    = p_j * (<dO[r,h], V[j,g]> - delta)
 *   dQ[r,h] = scale * sum_j dS_j K[j,g]
 *   dK[j,g] += scale * dS_j Q[r,h]        (over every listed r with j in vis(r), every h in g)
 *   dV[j,g] += p_j dO[r,h]
 *
 * Inputs Q, K, V, dO are bf16 bit patterns in compact-row layout ([N][H][D]); every value is
 * read exactly as a double.  lse is evaluated as max + ln(sum exp(s - max)), which is the
 * same quantity.  The loops run over rows (forward, dQ) and over disjoint ranges of key
 * rows (dK, dV) on plain POSIX threads; each output element is written by one thread only,
 * so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int64_t N, n_rows;
    int Hq, Hkv, D;
    double scale;
    const uint16_t *q, *k, *v, *dout;
    const int64_t *rows, *ptr, *lo, *hi;
    const double *o_in, *lse_in;        /* backward inputs (oracle forward results) */
    double *o, *lse, *delta, *dq, *dk, *dv;
    int64_t chunk;                      /* key rows per dK/dV task */
    int64_t next;                       /* work counter (atomic) */
    int64_t max_vis;
} job_t;

static double bf(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double dot_bf_bf(const uint16_t *a, const uint16_t *b, int D) {
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += bf(a[d]) * bf(b[d]);
    return s;
}

static double dot_bf_d(const uint16_t *a, const double *b, int D) {
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += bf(a[d]) * b[d];
    return s;
}

static int64_t take(job_t *J) { return __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED); }

/* ---------------------------------------------------------------- forward, per listed row */
static void *fwd_worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int G = J->Hq / J->Hkv, D = J->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->max_vis > 0 ? J->max_vis : 1));
    for (;;) {
        int64_t t = take(J);
        if (t >= J->n_rows) break;
        const int64_t r = J->rows[t];
        for (int h = 0; h < J->Hq; ++h) {
            const int g = h / G;
            const uint16_t *qr = J->q + ((size_t)r * J->Hq + h) * D;
            int64_t n = 0;
            double m = -INFINITY;
            for (int64_t e = J->ptr[t]; e < J->ptr[t + 1]; ++e)
                for (int64_t j = J->lo[e]; j < J->hi[e]; ++j) {
                    s[n] = J->scale * dot_bf_bf(qr, J->k + ((size_t)j * J->Hkv + g) * D, D);
                    if (s[n] > m) m = s[n];
                    ++n;
                }
            double l = 0.0;
            for (int64_t i = 0; i < n; ++i) l += exp(s[i] - m);
            const double lse = m + log(l);
            double *orow = J->o + ((size_t)t * J->Hq + h) * D;
            for (int d = 0; d < D; ++d) orow[d] = 0.0;
            n = 0;
            for (int64_t e = J->ptr[t]; e < J->ptr[t + 1]; ++e)
                for (int64_t j = J->lo[e]; j < J->hi[e]; ++j) {
                    const double p = exp(s[n++] - lse);
                    const uint16_t *vj = J->v + ((size_t)j * J->Hkv + g) * D;
                    for (int d = 0; d < D; ++d) orow[d] += p * bf(vj[d]);
                }
            J->lse[(size_t)t * J->Hq + h] = lse;
        }
    }
    free(s);
    return NULL;
}

/* --------------------------------------------------- backward part 1: delta and dQ per row */
static void *dq_worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int G = J->Hq / J->Hkv, D = J->D;
    for (;;) {
        int64_t t = take(J);
        if (t >= J->n_rows) break;
        const int64_t r = J->rows[t];
        for (int h = 0; h < J->Hq; ++h) {
            const int g = h / G;
            const uint16_t *qr = J->q + ((size_t)r * J->Hq + h) * D;
            const uint16_t *dor = J->dout + ((size_t)r * J->Hq + h) * D;
            const double *orow = J->o_in + ((size_t)t * J->Hq + h) * D;
            const double lse = J->lse_in[(size_t)t * J->Hq + h];
            const double delta = dot_bf_d(dor, orow, D);
            J->delta[(size_t)t * J->Hq + h] = delta;
            double *dqr = J->dq + ((size_t)t * J->Hq + h) * D;
            for (int d = 0; d < D; ++d) dqr[d] = 0.0;
            for (int64_t e = J->ptr[t]; e < J->ptr[t + 1]; ++e)
                for (int64_t j = J->lo[e]; j < J->hi[e]; ++j) {
                    const uint16_t *kj = J->k + ((size_t)j * J->Hkv + g) * D;
                    const uint16_t *vj = J->v + ((size_t)j * J->Hkv + g) * D;
                    const double p = exp(J->scale * dot_bf_bf(qr, kj, D) - lse);
                    const double ds = p * (dot_bf_bf(dor, vj, D) - delta);
                    for (int d = 0; d < D; ++d) dqr[d] += J->scale * ds * bf(kj[d]);
                }
        }
    }
    return NULL;
}

/* ------------------------------------- backward part 2: dK, dV over disjoint key-row ranges */
static void *dkdv_worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int G = J->Hq / J->Hkv, D = J->D;
    const int64_t n_tasks = (J->N + J->chunk - 1) / J->chunk;
    for (;;) {
        int64_t task = take(J);
        if (task >= n_tasks) break;
        const int64_t c0 = task * J->chunk, c1 = c0 + J->chunk < J->N ? c0 + J->chunk : J->N;
        for (int64_t t = 0; t < J->n_rows; ++t) {
            const int64_t r = J->rows[t];
            for (int64_t e = J->ptr[t]; e < J->ptr[t + 1]; ++e) {
                const int64_t lo = J->lo[e] > c0 ? J->lo[e] : c0;
                const int64_t hi = J->hi[e] < c1 ? J->hi[e] : c1;
                for (int64_t j = lo; j < hi; ++j)
                    for (int h = 0; h < J->Hq; ++h) {
                        const int g = h / G;
                        const uint16_t *qr = J->q + ((size_t)r * J->Hq + h) * D;
                        const uint16_t *dor = J->dout + ((size_t)r * J->Hq + h) * D;
                        const uint16_t *kj = J->k + ((size_t)j * J->Hkv + g) * D;
                        const uint16_t *vj = J->v + ((size_t)j * J->Hkv + g) * D;
                        const double lse = J->lse_in[(size_t)t * J->Hq + h];
                        const double delta = J->delta[(size_t)t * J->Hq + h];
                        const double p = exp(J->scale * dot_bf_bf(qr, kj, D) - lse);
                        const double ds = p * (dot_bf_bf(dor, vj, D) - delta);
                        double *dkj = J->dk + ((size_t)j * J->Hkv + g) * D;
                        double *dvj = J->dv + ((size_t)j * J->Hkv + g) * D;
                        for (int d = 0; d < D; ++d) {
                            dkj[d] += J->scale * ds * bf(qr[d]);
                            dvj[d] += p * bf(dor[d]);
                        }
                    }
            }
        }
    }
    return NULL;
}

static int run(job_t *J, void *(*fn)(void *), int n_threads) {
    if (n_threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = c > 0 ? (int)c : 1;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    J->next = 0;
    int started = 0;
    for (int i = 0; i < n_threads; ++i)
        if (pthread_create(&th[i], NULL, fn, J) == 0) ++started;
    if (started == 0) fn(J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return started > 0 ? started : 1;
}

static int64_t max_visible(const int64_t *ptr, const int64_t *lo, const int64_t *hi, int64_t n) {
    int64_t best = 0;
    for (int64_t t = 0; t < n; ++t) {
        int64_t c = 0;
        for (int64_t e = ptr[t]; e < ptr[t + 1]; ++e) c += hi[e] - lo[e];
        if (c > best) best = c;
    }
    return best;
}

/* Forward for the listed rows.  o: [n_rows][Hq][D], lse: [n_rows][Hq].
 * Returns the number of threads used. */
int oracle_forward(int64_t N, int Hq, int Hkv, int D, double scale,
                   const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   int64_t n_rows, const int64_t *rows, const int64_t *ptr,
                   const int64_t *lo, const int64_t *hi,
                   double *o, double *lse, int n_threads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.N = N; J.n_rows = n_rows; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.rows = rows; J.ptr = ptr; J.lo = lo; J.hi = hi;
    J.o = o; J.lse = lse;
    J.max_vis = max_visible(ptr, lo, hi, n_rows);
    return run(&J, fwd_worker, n_threads);
}

/* Backward for the listed rows, given the forward results o_in / lse_in of those rows.
 * delta: [n_rows][Hq]; dq: [n_rows][Hq][D]; dk, dv: [N][Hkv][D], written (not accumulated)
 * with the sum of the contributions of the listed rows.  Returns the thread count. */
int oracle_backward(int64_t N, int Hq, int Hkv, int D, double scale,
                    const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const uint16_t *dout, int64_t n_rows, const int64_t *rows,
                    const int64_t *ptr, const int64_t *lo, const int64_t *hi,
                    const double *o_in, const double *lse_in,
                    double *delta, double *dq, double *dk, double *dv, int n_threads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.N = N; J.n_rows = n_rows; J.Hq = Hq; J.Hkv = Hkv; J.D = D; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.dout = dout;
    J.rows = rows; J.ptr = ptr; J.lo = lo; J.hi = hi;
    J.o_in = o_in; J.lse_in = lse_in; J.delta = delta; J.dq = dq; J.dk = dk; J.dv = dv;
    int used = run(&J, dq_worker, n_threads);
    if (dk && dv) {
        memset(dk, 0, sizeof(double) * (size_t)N * Hkv * D);
        memset(dv, 0, sizeof(double) * (size_t)N * Hkv * D);
        J.chunk = 64;
        run(&J, dkdv_worker, n_threads);
    }
    return used;
}
