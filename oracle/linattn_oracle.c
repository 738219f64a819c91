/*
 * Float64 CPU oracle for kernelized linear attention with phi(x) = elu(x) + 1.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * CPU-baseline leg may load this library. The CUDA library never links it and
 * shares no code, header or constant with it.
 *
 * Every routine is the plain definition, written out in double precision with
 * no blocking, fusion or reordering beyond what the definition states:
 *
 *   phi(x) = x + 1 for x > 0, exp(x) for x <= 0
 *       ("Why Replace Attention? ..." blog, section 5.3, the boxed elu+1 map;
 *        "Transformers Are RNNs: Linear Attention" note, "Factor the
 *        Similarity Kernel").
 *   quadratic form: w_ij = phi(q_i).phi(k_j) over j <= i (causal) or all j,
 *       o_i = sum_j w_ij v_j / (sum_j w_ij + eps)
 *       ("Why Replace Attention? ..." sections 5.7 and 7.1; the worked
 *        similarity matrix of section 6.5).
 *   recurrent form: S_0 = 0, z_0 = 0; S_i = S_{i-1} + phi(k_i) v_i^T,
 *       z_i = z_{i-1} + phi(k_i); o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps)
 *       ("Why Replace Attention? ..." section 7.2, boxed recurrence;
 *        "Transformers Are RNNs: Linear Attention", "Turn Causal Attention
 *        into a Recurrence"). The non-causal output reads the final S, z for
 *        every row (same blog, section 6.2, boxed S, z and o_i).
 *   decode step: one iteration of the recurrence on caller-owned (S, z),
 *       update first, then read.
 *
 * eps is added once to the scalar denominator. The pages say only that an
 * epsilon is needed in practice ("Transformers Are RNNs: Linear Attention",
 * "Where It Breaks", ill-conditioned denominator); its value and placement
 * are this library's reading, with eps = 0 giving the exact printed form.
 *
 * Layout: q, k are [BH, N, D], v and o are [BH, N, M], S is [BH, D, M]
 * (row = feature index c, column = value index m), z is [BH, D]. All
 * row-major, contiguous, double.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

double ora_phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

void ora_phi_array(const double* x, double* y, long n)
{
    for (long i = 0; i < n; ++i) y[i] = ora_phi(x[i]);
}

/* ---------------------------------------------------------------- heads */

typedef struct {
    const double *q, *k, *v;
    double *o, *S_out, *z_out;
    long BH, N;
    int D, M, causal, form;
    double eps;
    long h_begin, h_end;
    int status;
} ora_job;

enum { FORM_QUADRATIC = 0, FORM_RECURRENT = 1 };

/* o_i = sum_j w_ij v_j / (sum_j w_ij + eps), w_ij = phi(q_i).phi(k_j). */
static int quadratic_head(const double* q, const double* k, const double* v, double* o,
                          long N, int D, int M, int causal, double eps)
{
    double* fk = (double*)malloc(sizeof(double) * (size_t)N * (size_t)D);
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    double* num = (double*)malloc(sizeof(double) * (size_t)M);
    if (!fk || !fq || !num) { free(fk); free(fq); free(num); return 1; }
    for (long j = 0; j < N; ++j)
        for (int c = 0; c < D; ++c) fk[j * D + c] = ora_phi(k[j * D + c]);
    for (long i = 0; i < N; ++i) {
        for (int c = 0; c < D; ++c) fq[c] = ora_phi(q[i * D + c]);
        for (int m = 0; m < M; ++m) num[m] = 0.0;
        double den = 0.0;
        long jend = causal ? i + 1 : N;
        for (long j = 0; j < jend; ++j) {
            double w = 0.0;
            for (int c = 0; c < D; ++c) w += fq[c] * fk[j * D + c];
            den += w;
            for (int m = 0; m < M; ++m) num[m] += w * v[j * M + m];
        }
        for (int m = 0; m < M; ++m) o[i * M + m] = num[m] / (den + eps);
    }
    free(fk); free(fq); free(num);
    return 0;
}

/* o_i = phi(q_i)^T S / (phi(q_i)^T z + eps) for one query row. */
static void read_state(const double* qi, const double* S, const double* z, double* oi,
                       int D, int M, double eps, double* fq)
{
    for (int c = 0; c < D; ++c) fq[c] = ora_phi(qi[c]);
    double den = 0.0;
    for (int c = 0; c < D; ++c) den += fq[c] * z[c];
    for (int m = 0; m < M; ++m) {
        double num = 0.0;
        for (int c = 0; c < D; ++c) num += fq[c] * S[c * M + m];
        oi[m] = num / (den + eps);
    }
}

/* S += phi(k_i) v_i^T, z += phi(k_i). */
static void update_state(const double* ki, const double* vi, double* S, double* z,
                         int D, int M, double* fk)
{
    for (int c = 0; c < D; ++c) fk[c] = ora_phi(ki[c]);
    for (int c = 0; c < D; ++c) {
        z[c] += fk[c];
        for (int m = 0; m < M; ++m) S[c * M + m] += fk[c] * vi[m];
    }
}

static int recurrent_head(const double* q, const double* k, const double* v, double* o,
                          double* S_out, double* z_out,
                          long N, int D, int M, int causal, double eps)
{
    double* S = (double*)calloc((size_t)D * (size_t)M, sizeof(double));
    double* z = (double*)calloc((size_t)D, sizeof(double));
    double* f = (double*)malloc(sizeof(double) * (size_t)D);
    if (!S || !z || !f) { free(S); free(z); free(f); return 1; }
    for (long i = 0; i < N; ++i) {
        update_state(k + i * D, v + i * M, S, z, D, M, f);
        if (causal) read_state(q + i * D, S, z, o + i * M, D, M, eps, f);
    }
    if (!causal)
        for (long i = 0; i < N; ++i) read_state(q + i * D, S, z, o + i * M, D, M, eps, f);
    if (S_out) memcpy(S_out, S, sizeof(double) * (size_t)D * (size_t)M);
    if (z_out) memcpy(z_out, z, sizeof(double) * (size_t)D);
    free(S); free(z); free(f);
    return 0;
}

static void* run_job(void* arg)
{
    ora_job* jb = (ora_job*)arg;
    jb->status = 0;
    for (long h = jb->h_begin; h < jb->h_end; ++h) {
        const double* q = jb->q + h * jb->N * jb->D;
        const double* k = jb->k + h * jb->N * jb->D;
        const double* v = jb->v + h * jb->N * jb->M;
        double* o = jb->o + h * jb->N * jb->M;
        int rc;
        if (jb->form == FORM_QUADRATIC) {
            rc = quadratic_head(q, k, v, o, jb->N, jb->D, jb->M, jb->causal, jb->eps);
        } else {
            double* So = jb->S_out ? jb->S_out + h * (long)jb->D * jb->M : NULL;
            double* zo = jb->z_out ? jb->z_out + h * (long)jb->D : NULL;
            rc = recurrent_head(q, k, v, o, So, zo, jb->N, jb->D, jb->M, jb->causal, jb->eps);
        }
        if (rc) { jb->status = rc; break; }
    }
    return NULL;
}

/* Splits the independent heads over nthreads POSIX threads. Returns 0 on success. */
static int run_heads(ora_job base, int nthreads)
{
    if (base.BH <= 0 || base.N < 0 || base.D <= 0 || base.M <= 0) return 2;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > base.BH) nthreads = (int)base.BH;
    ora_job* jobs = (ora_job*)malloc(sizeof(ora_job) * (size_t)nthreads);
    pthread_t* tids = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !tids) { free(jobs); free(tids); return 1; }
    long per = base.BH / nthreads, extra = base.BH % nthreads, h = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].h_begin = h;
        h += per + (t < extra ? 1 : 0);
        jobs[t].h_end = h;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_job, &jobs[t]) != 0) break;
        started = t;
    }
    run_job(&jobs[0]);
    /* Threads that failed to start are run here, in order. */
    for (int t = started + 1; t < nthreads; ++t) run_job(&jobs[t]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    int status = 0;
    for (int t = 0; t < nthreads; ++t) if (jobs[t].status) status = jobs[t].status;
    free(jobs); free(tids);
    return status;
}

int ora_quadratic(const double* q, const double* k, const double* v, double* o,
                  long BH, long N, int D, int M, int causal, double eps, int nthreads)
{
    ora_job b = {q, k, v, o, NULL, NULL, BH, N, D, M, causal, FORM_QUADRATIC, eps, 0, 0, 0};
    return run_heads(b, nthreads);
}

int ora_recurrent(const double* q, const double* k, const double* v, double* o,
                  double* S_out, double* z_out,
                  long BH, long N, int D, int M, int causal, double eps, int nthreads)
{
    ora_job b = {q, k, v, o, S_out, z_out, BH, N, D, M, causal, FORM_RECURRENT, eps, 0, 0, 0};
    return run_heads(b, nthreads);
}

/*
 * One token of the recurrence per head, on caller state: S <- S + phi(k) v^T,
 * z <- z + phi(k), then o = phi(q)^T S / (phi(q)^T z + eps).
 * q, k are [BH, D]; v, o are [BH, M]; S is [BH, D, M]; z is [BH, D].
 */
int ora_decode_step(const double* q, const double* k, const double* v, double* o,
                    double* S, double* z, long BH, int D, int M, double eps)
{
    if (BH <= 0 || D <= 0 || M <= 0) return 2;
    double* f = (double*)malloc(sizeof(double) * (size_t)D);
    if (!f) return 1;
    for (long h = 0; h < BH; ++h) {
        double* Sh = S + h * (long)D * M;
        double* zh = z + h * (long)D;
        update_state(k + h * D, v + h * M, Sh, zh, D, M, f);
        read_state(q + h * D, Sh, zh, o + h * M, D, M, eps, f);
    }
    free(f);
    return 0;
}

/*
 * Selected output rows by the quadratic definition, for spot checks of large
 * problems: for each r, row (heads[r], rows[r]) of o is written to out[r*M..].
 */
int ora_rows(const double* q, const double* k, const double* v,
             long BH, long N, int D, int M, int causal, double eps,
             const long* heads, const long* rows, long nsel, double* out)
{
    double* fq = (double*)malloc(sizeof(double) * (size_t)D);
    double* num = (double*)malloc(sizeof(double) * (size_t)M);
    if (!fq || !num) { free(fq); free(num); return 1; }
    for (long r = 0; r < nsel; ++r) {
        long h = heads[r], i = rows[r];
        if (h < 0 || h >= BH || i < 0 || i >= N) { free(fq); free(num); return 2; }
        const double* qh = q + h * N * D;
        const double* kh = k + h * N * D;
        const double* vh = v + h * N * M;
        for (int c = 0; c < D; ++c) fq[c] = ora_phi(qh[i * D + c]);
        for (int m = 0; m < M; ++m) num[m] = 0.0;
        double den = 0.0;
        long jend = causal ? i + 1 : N;
        for (long j = 0; j < jend; ++j) {
            double w = 0.0;
            for (int c = 0; c < D; ++c) w += fq[c] * ora_phi(kh[j * D + c]);
            den += w;
            for (int m = 0; m < M; ++m) num[m] += w * vh[j * M + m];
        }
        for (int m = 0; m < M; ++m) out[r * M + m] = num[m] / (den + eps);
    }
    free(fq); free(num);
    return 0;
}
