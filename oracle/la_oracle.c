/*
 * la_oracle.c -- plain fp64 CPU oracle for kernelized linear attention.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the bench's
 * CPU baseline leg; never by the product path.  Each routine writes out the
 * definition it cites with no blocking, fusion or reordering beyond it.
 * See la_oracle.h for layouts.
 */
#define _GNU_SOURCE
#include "la_oracle.h"

#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* elu(x) = x for x > 0, alpha (e^x - 1) otherwise, alpha = 1.0
 * ("Transformers are RNNs", section 特征映射, eq. elu); phi = elu + 1. */
static const double ELU_ALPHA = 1.0;

double lao_phi(double x) {
    /* x <= 0: alpha (e^x - 1) + 1, written as alpha e^x + (1 - alpha) so that
     * it does not cancel to 0 for very negative x (it is e^x for alpha = 1). */
    return x > 0.0 ? x + 1.0 : ELU_ALPHA * exp(x) + (1.0 - ELU_ALPHA);
}

/* d/dx of elu(x) + 1: 1 for x > 0, alpha e^x otherwise (continuous at 0). */
double lao_dphi(double x) { return x > 0.0 ? 1.0 : ELU_ALPHA * exp(x); }

int lao_default_threads(void) {
    cpu_set_t set;
    CPU_ZERO(&set);
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ---------------------------------------------------------------- helpers */

static double* phi_rows(const double* X, int N, int D) {
    double* out = (double*)malloc(sizeof(double) * (size_t)N * (size_t)D);
    for (size_t t = 0; t < (size_t)N * (size_t)D; ++t) out[t] = lao_phi(X[t]);
    return out;
}

static double dot(const double* a, const double* b, int n) {
    double s = 0.0;
    for (int t = 0; t < n; ++t) s += a[t] * b[t];
    return s;
}

/* Runs fn(h, ctx) for h in [0, nh) on up to nthreads host threads. */
typedef void (*head_fn)(int h, void* ctx);
typedef struct {
    head_fn fn;
    void* ctx;
    int h0, h1;
} span_t;

static void* run_span(void* p) {
    span_t* s = (span_t*)p;
    for (int h = s->h0; h < s->h1; ++h) s->fn(h, s->ctx);
    return NULL;
}

static void for_heads(int nh, int nthreads, head_fn fn, void* ctx) {
    if (nthreads <= 0) nthreads = lao_default_threads();
    if (nthreads > nh) nthreads = nh;
    if (nthreads <= 1) {
        for (int h = 0; h < nh; ++h) fn(h, ctx);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    span_t* sp = (span_t*)malloc(sizeof(span_t) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        sp[t].fn = fn;
        sp[t].ctx = ctx;
        sp[t].h0 = (int)((long)nh * t / nthreads);
        sp[t].h1 = (int)((long)nh * (t + 1) / nthreads);
        pthread_create(&th[t], NULL, run_span, &sp[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(sp);
}

/* ------------------------------------------------- forward, quadratic forms */

/* Generalised attention with sim(q, k) = phi(q).phi(k): section 二 eq. common
 * and the kernelised numerator/denominator; causal when `causal` (section 三
 * eq. mask, j <= i). */
static void quadratic_forward(int nh, int N, int D, int M, const double* Q, const double* K,
                              const double* V, double* O, int causal) {
    double* num = (double*)malloc(sizeof(double) * (size_t)M);
    for (int h = 0; h < nh; ++h) {
        const double* Qh = Q + (size_t)h * N * D;
        const double* Kh = K + (size_t)h * N * D;
        const double* Vh = V + (size_t)h * N * M;
        double* Oh = O + (size_t)h * N * M;
        double* fq = phi_rows(Qh, N, D);
        double* fk = phi_rows(Kh, N, D);
        for (int i = 0; i < N; ++i) {
            int jmax = causal ? i : N - 1;
            double den = 0.0;
            memset(num, 0, sizeof(double) * (size_t)M);
            for (int j = 0; j <= jmax; ++j) {
                double w = dot(fq + (size_t)i * D, fk + (size_t)j * D, D);
                den += w;
                for (int e = 0; e < M; ++e) num[e] += w * Vh[(size_t)j * M + e];
            }
            for (int e = 0; e < M; ++e) Oh[(size_t)i * M + e] = num[e] / den;
        }
        free(fq);
        free(fk);
    }
    free(num);
}

void lao_causal_forward_quadratic(int nh, int N, int D, int M, const double* Q,
                                  const double* K, const double* V, double* O) {
    quadratic_forward(nh, N, D, M, Q, K, V, O, 1);
}

void lao_noncausal_forward_quadratic(int nh, int N, int D, int M, const double* Q,
                                     const double* K, const double* V, double* O) {
    quadratic_forward(nh, N, D, M, Q, K, V, O, 0);
}

/* ------------------------------------------------- forward, recurrent form */

typedef struct {
    int N, D, M;
    const double *Q, *K, *V, *S0, *Z0;
    double *O, *S_out, *Z_out, *den_out;
} rec_ctx;

/* Section 三: S_t = S_{t-1} + phi(K_t) V_t^T, Z_t = Z_{t-1} + phi(K_t), then
 * eq. output V'_t = phi(Q_t)^T S_t / phi(Q_t)^T Z_t; the denominator
 * phi(Q_t)^T Z_t is also returned per token when den_out is given. */
static void recurrent_head(int h, void* p) {
    rec_ctx* c = (rec_ctx*)p;
    const int N = c->N, D = c->D, M = c->M;
    const double* Qh = c->Q + (size_t)h * N * D;
    const double* Kh = c->K + (size_t)h * N * D;
    const double* Vh = c->V + (size_t)h * N * M;
    double* Oh = c->O + (size_t)h * N * M;
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* kf = (double*)malloc(sizeof(double) * (size_t)D);
    double* qf = (double*)malloc(sizeof(double) * (size_t)D);
    if (c->S0) memcpy(S, c->S0 + (size_t)h * D * M, sizeof(double) * (size_t)D * M);
    if (c->Z0) memcpy(Z, c->Z0 + (size_t)h * D, sizeof(double) * (size_t)D);
    for (int t = 0; t < N; ++t) {
        const double* vt = Vh + (size_t)t * M;
        for (int d = 0; d < D; ++d) kf[d] = lao_phi(Kh[(size_t)t * D + d]);
        for (int d = 0; d < D; ++d) {
            for (int e = 0; e < M; ++e) S[(size_t)d * M + e] += kf[d] * vt[e];
            Z[d] += kf[d];
        }
        for (int d = 0; d < D; ++d) qf[d] = lao_phi(Qh[(size_t)t * D + d]);
        double den = dot(qf, Z, D);
        if (c->den_out) c->den_out[(size_t)h * N + t] = den;
        for (int e = 0; e < M; ++e) {
            double num = 0.0;
            for (int d = 0; d < D; ++d) num += qf[d] * S[(size_t)d * M + e];
            Oh[(size_t)t * M + e] = num / den;
        }
    }
    if (c->S_out) memcpy(c->S_out + (size_t)h * D * M, S, sizeof(double) * (size_t)D * M);
    if (c->Z_out) memcpy(c->Z_out + (size_t)h * D, Z, sizeof(double) * (size_t)D);
    free(S);
    free(Z);
    free(kf);
    free(qf);
}

void lao_causal_forward_recurrent(int nh, int N, int D, int M, const double* Q,
                                  const double* K, const double* V,
                                  const double* S0, const double* Z0, double* O,
                                  double* S_out, double* Z_out, double* den_out, int nthreads) {
    rec_ctx c = {N, D, M, Q, K, V, S0, Z0, O, S_out, Z_out, den_out};
    for_heads(nh, nthreads, recurrent_head, &c);
}

/* ------------------------------------------ non-causal, associativity form */

typedef struct {
    int N, D, M;
    const double *Q, *K, *V;
    double *O, *S_out, *Z_out;
} assoc_ctx;

/* Section 二 eq. linear: S = sum_j phi(K_j) V_j^T and Z = sum_j phi(K_j) are
 * formed once, then reused for every query. */
static void assoc_head(int h, void* p) {
    assoc_ctx* c = (assoc_ctx*)p;
    const int N = c->N, D = c->D, M = c->M;
    const double* Qh = c->Q + (size_t)h * N * D;
    const double* Kh = c->K + (size_t)h * N * D;
    const double* Vh = c->V + (size_t)h * N * M;
    double* Oh = c->O + (size_t)h * N * M;
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* f = (double*)malloc(sizeof(double) * (size_t)D);
    for (int j = 0; j < N; ++j) {
        for (int d = 0; d < D; ++d) f[d] = lao_phi(Kh[(size_t)j * D + d]);
        for (int d = 0; d < D; ++d) {
            for (int e = 0; e < M; ++e) S[(size_t)d * M + e] += f[d] * Vh[(size_t)j * M + e];
            Z[d] += f[d];
        }
    }
    for (int i = 0; i < N; ++i) {
        for (int d = 0; d < D; ++d) f[d] = lao_phi(Qh[(size_t)i * D + d]);
        double den = dot(f, Z, D);
        for (int e = 0; e < M; ++e) {
            double num = 0.0;
            for (int d = 0; d < D; ++d) num += f[d] * S[(size_t)d * M + e];
            Oh[(size_t)i * M + e] = num / den;
        }
    }
    if (c->S_out) memcpy(c->S_out + (size_t)h * D * M, S, sizeof(double) * (size_t)D * M);
    if (c->Z_out) memcpy(c->Z_out + (size_t)h * D, Z, sizeof(double) * (size_t)D);
    free(S);
    free(Z);
    free(f);
}

void lao_noncausal_forward_assoc(int nh, int N, int D, int M, const double* Q,
                                 const double* K, const double* V, double* O,
                                 double* S_out, double* Z_out, int nthreads) {
    assoc_ctx c = {N, D, M, Q, K, V, O, S_out, Z_out};
    for_heads(nh, nthreads, assoc_head, &c);
}

/* ------------------------------------------- backward, cumulative-sum form */

typedef struct {
    int N, D, M;
    const double *Q, *K, *V, *G;
    double *dQ, *dK, *dV;
} bwd_ctx;

/*
 * With qf = phi(Q), kf = phi(K), den_i = qf_i.Z_i and O_i = qf_i^T S_i / den_i:
 *   gn_i = G_i / den_i          (gradient reaching the numerator of row i)
 *   gd_i = -(G_i . O_i) / den_i (gradient reaching the denominator of row i)
 * The denominator is the numerator with V replaced by ones; the pages leave its
 * gradient to autograd ("Transformers are RNNs" section 三（一）), and the
 * quotient rule gives the two lines above.  Then, eqs. gq-gv of section
 * 三（一）4 extended by the denominator term:
 *   dqf_i = S_i gn_i + Z_i gd_i                  (prefix state S_i, Z_i)
 *   R_i = sum_{j>=i} qf_j gn_j^T, r_i = sum_{j>=i} qf_j gd_j   (suffix state)
 *   dkf_i = R_i V_i + r_i,   dV_i = R_i^T kf_i
 * and finally dQ = dqf * phi'(Q), dK = dkf * phi'(K).
 */
static void bwd_cumsum_head(int h, void* p) {
    bwd_ctx* c = (bwd_ctx*)p;
    const int N = c->N, D = c->D, M = c->M;
    const double* Qh = c->Q + (size_t)h * N * D;
    const double* Kh = c->K + (size_t)h * N * D;
    const double* Vh = c->V + (size_t)h * N * M;
    const double* Gh = c->G + (size_t)h * N * M;
    double* dQh = c->dQ + (size_t)h * N * D;
    double* dKh = c->dK + (size_t)h * N * D;
    double* dVh = c->dV + (size_t)h * N * M;

    double* qf = phi_rows(Qh, N, D);
    double* kf = phi_rows(Kh, N, D);
    double* gn = (double*)malloc(sizeof(double) * (size_t)N * M);
    double* gd = (double*)malloc(sizeof(double) * (size_t)N);
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* o = (double*)malloc(sizeof(double) * (size_t)M);

    /* prefix direction: S_i, Z_i include token i */
    for (int i = 0; i < N; ++i) {
        const double* ki = kf + (size_t)i * D;
        const double* vi = Vh + (size_t)i * M;
        const double* qi = qf + (size_t)i * D;
        for (int d = 0; d < D; ++d) {
            for (int e = 0; e < M; ++e) S[(size_t)d * M + e] += ki[d] * vi[e];
            Z[d] += ki[d];
        }
        double den = dot(qi, Z, D);
        for (int e = 0; e < M; ++e) {
            double num = 0.0;
            for (int d = 0; d < D; ++d) num += qi[d] * S[(size_t)d * M + e];
            o[e] = num / den;
        }
        const double* gi = Gh + (size_t)i * M;
        double go = dot(gi, o, M);
        for (int e = 0; e < M; ++e) gn[(size_t)i * M + e] = gi[e] / den;
        gd[i] = -go / den;
        for (int d = 0; d < D; ++d) {
            double acc = Z[d] * gd[i];
            for (int e = 0; e < M; ++e) acc += S[(size_t)d * M + e] * gn[(size_t)i * M + e];
            dQh[(size_t)i * D + d] = acc * lao_dphi(Qh[(size_t)i * D + d]);
        }
    }

    /* suffix direction: R_i, r_i include token i */
    double* R = S; /* reuse storage */
    double* r = Z;
    memset(R, 0, sizeof(double) * (size_t)D * M);
    memset(r, 0, sizeof(double) * (size_t)D);
    for (int i = N - 1; i >= 0; --i) {
        const double* qi = qf + (size_t)i * D;
        const double* gni = gn + (size_t)i * M;
        for (int d = 0; d < D; ++d) {
            for (int e = 0; e < M; ++e) R[(size_t)d * M + e] += qi[d] * gni[e];
            r[d] += qi[d] * gd[i];
        }
        const double* ki = kf + (size_t)i * D;
        const double* vi = Vh + (size_t)i * M;
        for (int d = 0; d < D; ++d) {
            double acc = r[d];
            for (int e = 0; e < M; ++e) acc += R[(size_t)d * M + e] * vi[e];
            dKh[(size_t)i * D + d] = acc * lao_dphi(Kh[(size_t)i * D + d]);
        }
        for (int e = 0; e < M; ++e) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += R[(size_t)d * M + e] * ki[d];
            dVh[(size_t)i * M + e] = acc;
        }
    }
    free(qf);
    free(kf);
    free(gn);
    free(gd);
    free(S);
    free(Z);
    free(o);
}

void lao_causal_backward_cumsum(int nh, int N, int D, int M, const double* Q,
                                const double* K, const double* V, const double* G,
                                double* dQ, double* dK, double* dV, int nthreads) {
    bwd_ctx c = {N, D, M, Q, K, V, G, dQ, dK, dV};
    for_heads(nh, nthreads, bwd_cumsum_head, &c);
}

/* ----------------------------------------------- backward, quadratic form */

/*
 * Derivative of O_i = sum_{j<=i} w_ij V_j / sum_{j<=i} w_ij with
 * w_ij = qf_i.kf_j, taken term by term:
 *   dL/dw_ij = gn_i.V_j + gd_i            (j <= i)
 *   dqf_i = sum_{j<=i} dL/dw_ij kf_j,  dkf_j = sum_{i>=j} dL/dw_ij qf_i,
 *   dV_j  = sum_{i>=j} w_ij gn_i.
 */
void lao_causal_backward_quadratic(int nh, int N, int D, int M, const double* Q,
                                   const double* K, const double* V, const double* G,
                                   double* dQ, double* dK, double* dV) {
    for (int h = 0; h < nh; ++h) {
        const double* Qh = Q + (size_t)h * N * D;
        const double* Kh = K + (size_t)h * N * D;
        const double* Vh = V + (size_t)h * N * M;
        const double* Gh = G + (size_t)h * N * M;
        double* dQh = dQ + (size_t)h * N * D;
        double* dKh = dK + (size_t)h * N * D;
        double* dVh = dV + (size_t)h * N * M;
        double* qf = phi_rows(Qh, N, D);
        double* kf = phi_rows(Kh, N, D);
        double* w = (double*)calloc((size_t)N * N, sizeof(double));
        double* gn = (double*)malloc(sizeof(double) * (size_t)N * M);
        double* gd = (double*)malloc(sizeof(double) * (size_t)N);
        double* dqf = (double*)calloc((size_t)N * D, sizeof(double));
        double* dkf = (double*)calloc((size_t)N * D, sizeof(double));
        double* o = (double*)malloc(sizeof(double) * (size_t)M);
        memset(dVh, 0, sizeof(double) * (size_t)N * M);

        for (int i = 0; i < N; ++i) {
            double den = 0.0;
            for (int e = 0; e < M; ++e) o[e] = 0.0;
            for (int j = 0; j <= i; ++j) {
                double wij = dot(qf + (size_t)i * D, kf + (size_t)j * D, D);
                w[(size_t)i * N + j] = wij;
                den += wij;
                for (int e = 0; e < M; ++e) o[e] += wij * Vh[(size_t)j * M + e];
            }
            for (int e = 0; e < M; ++e) o[e] /= den;
            const double* gi = Gh + (size_t)i * M;
            for (int e = 0; e < M; ++e) gn[(size_t)i * M + e] = gi[e] / den;
            gd[i] = -dot(gi, o, M) / den;
        }
        for (int i = 0; i < N; ++i) {
            for (int j = 0; j <= i; ++j) {
                double dw = dot(gn + (size_t)i * M, Vh + (size_t)j * M, M) + gd[i];
                for (int d = 0; d < D; ++d) {
                    dqf[(size_t)i * D + d] += dw * kf[(size_t)j * D + d];
                    dkf[(size_t)j * D + d] += dw * qf[(size_t)i * D + d];
                }
                double wij = w[(size_t)i * N + j];
                for (int e = 0; e < M; ++e) dVh[(size_t)j * M + e] += wij * gn[(size_t)i * M + e];
            }
        }
        for (size_t t = 0; t < (size_t)N * D; ++t) {
            dQh[t] = dqf[t] * lao_dphi(Qh[t]);
            dKh[t] = dkf[t] * lao_dphi(Kh[t]);
        }
        free(qf);
        free(kf);
        free(w);
        free(gn);
        free(gd);
        free(dqf);
        free(dkf);
        free(o);
    }
}

/* ----------------------------------------- non-causal backward, state form */

typedef struct {
    int N, D, M;
    const double *Q, *K, *V, *G;
    double *dQ, *dK, *dV;
} ncb_ctx;

/*
 * Gradient of L = sum G * O for the non-causal form ("Transformers are RNNs"
 * section 二, eq. linear): the numerator gradients of section 三（一）4
 * (eqs. gq-gv) with the prefix state S_i and the suffix state R_i both taken
 * over every token, and the denominator by the quotient rule as in the causal
 * case:
 *   S = sum_j kf_j V_j^T, Z = sum_j kf_j, den_i = qf_i.Z, O_i = qf_i^T S / den_i
 *   gn_i = G_i / den_i,  gd_i = -(G_i . O_i) / den_i
 *   dqf_i = S gn_i + Z gd_i
 *   R = sum_i qf_i gn_i^T,  r = sum_i qf_i gd_i
 *   dkf_j = R V_j + r,  dV_j = R^T kf_j
 * then dQ = dqf * phi'(Q), dK = dkf * phi'(K).
 */
static void ncb_state_head(int h, void* p) {
    ncb_ctx* c = (ncb_ctx*)p;
    const int N = c->N, D = c->D, M = c->M;
    const double* Qh = c->Q + (size_t)h * N * D;
    const double* Kh = c->K + (size_t)h * N * D;
    const double* Vh = c->V + (size_t)h * N * M;
    const double* Gh = c->G + (size_t)h * N * M;
    double* dQh = c->dQ + (size_t)h * N * D;
    double* dKh = c->dK + (size_t)h * N * D;
    double* dVh = c->dV + (size_t)h * N * M;
    double* qf = phi_rows(Qh, N, D);
    double* kf = phi_rows(Kh, N, D);
    double* S = (double*)calloc((size_t)D * M, sizeof(double));
    double* Z = (double*)calloc((size_t)D, sizeof(double));
    double* R = (double*)calloc((size_t)D * M, sizeof(double));
    double* r = (double*)calloc((size_t)D, sizeof(double));
    double* gn = (double*)malloc(sizeof(double) * (size_t)M);
    double* o = (double*)malloc(sizeof(double) * (size_t)M);
    for (int j = 0; j < N; ++j) {
        const double* kj = kf + (size_t)j * D;
        for (int d = 0; d < D; ++d) {
            for (int e = 0; e < M; ++e) S[(size_t)d * M + e] += kj[d] * Vh[(size_t)j * M + e];
            Z[d] += kj[d];
        }
    }
    for (int i = 0; i < N; ++i) {
        const double* qi = qf + (size_t)i * D;
        const double* gi = Gh + (size_t)i * M;
        double den = dot(qi, Z, D);
        for (int e = 0; e < M; ++e) {
            double num = 0.0;
            for (int d = 0; d < D; ++d) num += qi[d] * S[(size_t)d * M + e];
            o[e] = num / den;
        }
        for (int e = 0; e < M; ++e) gn[e] = gi[e] / den;
        double gd = -dot(gi, o, M) / den;
        for (int d = 0; d < D; ++d) {
            double acc = Z[d] * gd;
            for (int e = 0; e < M; ++e) acc += S[(size_t)d * M + e] * gn[e];
            dQh[(size_t)i * D + d] = acc * lao_dphi(Qh[(size_t)i * D + d]);
            for (int e = 0; e < M; ++e) R[(size_t)d * M + e] += qi[d] * gn[e];
            r[d] += qi[d] * gd;
        }
    }
    for (int j = 0; j < N; ++j) {
        const double* kj = kf + (size_t)j * D;
        const double* vj = Vh + (size_t)j * M;
        for (int d = 0; d < D; ++d) {
            double acc = r[d];
            for (int e = 0; e < M; ++e) acc += R[(size_t)d * M + e] * vj[e];
            dKh[(size_t)j * D + d] = acc * lao_dphi(Kh[(size_t)j * D + d]);
        }
        for (int e = 0; e < M; ++e) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += R[(size_t)d * M + e] * kj[d];
            dVh[(size_t)j * M + e] = acc;
        }
    }
    free(qf);
    free(kf);
    free(S);
    free(Z);
    free(R);
    free(r);
    free(gn);
    free(o);
}

void lao_noncausal_backward_assoc(int nh, int N, int D, int M, const double* Q,
                                  const double* K, const double* V, const double* G,
                                  double* dQ, double* dK, double* dV, int nthreads) {
    ncb_ctx c = {N, D, M, Q, K, V, G, dQ, dK, dV};
    for_heads(nh, nthreads, ncb_state_head, &c);
}

/*
 * The same gradient from the unmasked quotient O_i = sum_j w_ij V_j / sum_j w_ij,
 * w_ij = qf_i.kf_j, term by term:
 *   dL/dw_ij = gn_i.V_j + gd_i   (every i, j)
 *   dqf_i = sum_j dL/dw_ij kf_j,  dkf_j = sum_i dL/dw_ij qf_i,  dV_j = sum_i w_ij gn_i.
 */
void lao_noncausal_backward_quadratic(int nh, int N, int D, int M, const double* Q,
                                      const double* K, const double* V, const double* G,
                                      double* dQ, double* dK, double* dV) {
    for (int h = 0; h < nh; ++h) {
        const double* Qh = Q + (size_t)h * N * D;
        const double* Kh = K + (size_t)h * N * D;
        const double* Vh = V + (size_t)h * N * M;
        const double* Gh = G + (size_t)h * N * M;
        double* dQh = dQ + (size_t)h * N * D;
        double* dKh = dK + (size_t)h * N * D;
        double* dVh = dV + (size_t)h * N * M;
        double* qf = phi_rows(Qh, N, D);
        double* kf = phi_rows(Kh, N, D);
        double* gn = (double*)malloc(sizeof(double) * (size_t)N * M);
        double* gd = (double*)malloc(sizeof(double) * (size_t)N);
        double* dqf = (double*)calloc((size_t)N * D, sizeof(double));
        double* dkf = (double*)calloc((size_t)N * D, sizeof(double));
        double* o = (double*)malloc(sizeof(double) * (size_t)M);
        memset(dVh, 0, sizeof(double) * (size_t)N * M);
        for (int i = 0; i < N; ++i) {
            double den = 0.0;
            for (int e = 0; e < M; ++e) o[e] = 0.0;
            for (int j = 0; j < N; ++j) {
                double wij = dot(qf + (size_t)i * D, kf + (size_t)j * D, D);
                den += wij;
                for (int e = 0; e < M; ++e) o[e] += wij * Vh[(size_t)j * M + e];
            }
            for (int e = 0; e < M; ++e) o[e] /= den;
            const double* gi = Gh + (size_t)i * M;
            for (int e = 0; e < M; ++e) gn[(size_t)i * M + e] = gi[e] / den;
            gd[i] = -dot(gi, o, M) / den;
        }
        for (int i = 0; i < N; ++i) {
            for (int j = 0; j < N; ++j) {
                double dw = dot(gn + (size_t)i * M, Vh + (size_t)j * M, M) + gd[i];
                double wij = dot(qf + (size_t)i * D, kf + (size_t)j * D, D);
                for (int d = 0; d < D; ++d) {
                    dqf[(size_t)i * D + d] += dw * kf[(size_t)j * D + d];
                    dkf[(size_t)j * D + d] += dw * qf[(size_t)i * D + d];
                }
                for (int e = 0; e < M; ++e) dVh[(size_t)j * M + e] += wij * gn[(size_t)i * M + e];
            }
        }
        for (size_t t = 0; t < (size_t)N * D; ++t) {
            dQh[t] = dqf[t] * lao_dphi(Qh[t]);
            dKh[t] = dkf[t] * lao_dphi(Kh[t]);
        }
        free(qf);
        free(kf);
        free(gn);
        free(gd);
        free(dqf);
        free(dkf);
        free(o);
    }
}

/* ------------------------------------------------------------ decode step */

/* RNN-mode inference ("Transformer与RNN的深层联结" section 2; "Transformers are
 * RNNs" section 四): first s += phi(k) v^T, z += phi(k), then read
 * phi(q)^T s / phi(q)^T z. */
void lao_decode_step(int nh, int D, int M, const double* q, const double* k,
                     const double* v, double* S, double* Z, double* out) {
    double* kf = (double*)malloc(sizeof(double) * (size_t)D);
    double* qf = (double*)malloc(sizeof(double) * (size_t)D);
    for (int h = 0; h < nh; ++h) {
        double* Sh = S + (size_t)h * D * M;
        double* Zh = Z + (size_t)h * D;
        const double* vh = v + (size_t)h * M;
        for (int d = 0; d < D; ++d) kf[d] = lao_phi(k[(size_t)h * D + d]);
        for (int d = 0; d < D; ++d) qf[d] = lao_phi(q[(size_t)h * D + d]);
        for (int d = 0; d < D; ++d) {
            for (int e = 0; e < M; ++e) Sh[(size_t)d * M + e] += kf[d] * vh[e];
            Zh[d] += kf[d];
        }
        double den = dot(qf, Zh, D);
        for (int e = 0; e < M; ++e) {
            double num = 0.0;
            for (int d = 0; d < D; ++d) num += qf[d] * Sh[(size_t)d * M + e];
            out[(size_t)h * M + e] = num / den;
        }
    }
    free(kf);
    free(qf);
}

/* ------------------------------------------- softmax KV-cache decode step */

/* Standard Transformer inference with a KV cache ("Transformer与RNN的深层联结"
 * section 2): the step's k, v are appended to the cache, then the query
 * attends to every cached position with softmax(q K^T / sqrt(D)) V (the
 * scaled dot-product of "Transformers are RNNs" section 一, eq. softmax).
 * Kc [nh][T][D], Vc [nh][T][M] hold the T earlier positions and are not
 * modified; the appended row is k [nh][D], v [nh][M].  The largest score is
 * subtracted before the exponentials (the pages' overflow guard, which does
 * not change the result). */
void lao_softmax_decode_step(int nh, int T, int D, int M, const double* q, const double* k,
                             const double* v, const double* Kc, const double* Vc, double* out) {
    double* sc = (double*)malloc(sizeof(double) * (size_t)(T + 1));
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
    for (int h = 0; h < nh; ++h) {
        const double* qh = q + (size_t)h * D;
        double mx = -INFINITY;
        for (int j = 0; j <= T; ++j) {
            const double* kj = j < T ? Kc + ((size_t)h * T + j) * D : k + (size_t)h * D;
            sc[j] = dot(qh, kj, D) * inv_sqrt_d;
            if (sc[j] > mx) mx = sc[j];
        }
        double den = 0.0;
        for (int j = 0; j <= T; ++j) {
            sc[j] = exp(sc[j] - mx);
            den += sc[j];
        }
        for (int e = 0; e < M; ++e) {
            double acc = 0.0;
            for (int j = 0; j <= T; ++j) {
                const double* vj = j < T ? Vc + ((size_t)h * T + j) * M : v + (size_t)h * M;
                acc += sc[j] * vj[e];
            }
            out[(size_t)h * M + e] = acc / den;
        }
    }
    free(sc);
}

/* ----------------------------------------------------- retention (decay) */

/* Decay of token t of head h: gates[h][t] when given (gated retention),
 * else gamma_head[h % H] (RetNet, one decay per head), else 1 (linear
 * attention without reflection).  `h` counts B*H heads, head index h % H. */
static double decay_of(int h, int t, int N, int H, const double* gamma_head, const double* gates) {
    if (gates) return gates[(size_t)h * N + t];
    if (gamma_head) return gamma_head[h % H];
    return 1.0;
}

/* "Transformer and Variants" section 1.3.2 (linear attention as an RNN without
 * the reflection term) and section 1.3.4 (RetNet, gated retention), in the
 * S = sum k v^T convention used throughout (S is the page's H transposed):
 *   S_t = gamma_t S_{t-1} + k_t v_t^T,   y_t = S_t^T q_t
 * raw q and k (no feature map) and no normaliser.  S0 (nullable) is the state
 * before token 0, S_out (nullable) receives the state after the last token. */
void lao_retention_forward_recurrent(int nh, int H, int N, int D, int M, const double* Q,
                                     const double* K, const double* V, const double* gamma_head,
                                     const double* gates, const double* S0, double* O,
                                     double* S_out) {
    double* S = (double*)malloc(sizeof(double) * (size_t)D * M);
    for (int h = 0; h < nh; ++h) {
        const double* Qh = Q + (size_t)h * N * D;
        const double* Kh = K + (size_t)h * N * D;
        const double* Vh = V + (size_t)h * N * M;
        double* Oh = O + (size_t)h * N * M;
        if (S0) memcpy(S, S0 + (size_t)h * D * M, sizeof(double) * (size_t)D * M);
        else memset(S, 0, sizeof(double) * (size_t)D * M);
        for (int t = 0; t < N; ++t) {
            const double g = decay_of(h, t, N, H, gamma_head, gates);
            for (int d = 0; d < D; ++d)
                for (int e = 0; e < M; ++e)
                    S[(size_t)d * M + e] = g * S[(size_t)d * M + e] +
                                           Kh[(size_t)t * D + d] * Vh[(size_t)t * M + e];
            for (int e = 0; e < M; ++e) {
                double y = 0.0;
                for (int d = 0; d < D; ++d) y += S[(size_t)d * M + e] * Qh[(size_t)t * D + d];
                Oh[(size_t)t * M + e] = y;
            }
        }
        if (S_out) memcpy(S_out + (size_t)h * D * M, S, sizeof(double) * (size_t)D * M);
    }
    free(S);
}

/* The same output unrolled (section 1.3.1's expansion of y_t as a sum over
 * j <= t, with the decays of the later tokens multiplied in):
 *   y_t = sum_{j<=t} (prod_{l=j+1..t} gamma_l) (k_j . q_t) v_j
 * (no initial state). */
void lao_retention_forward_quadratic(int nh, int H, int N, int D, int M, const double* Q,
                                     const double* K, const double* V, const double* gamma_head,
                                     const double* gates, double* O) {
    for (int h = 0; h < nh; ++h) {
        const double* Qh = Q + (size_t)h * N * D;
        const double* Kh = K + (size_t)h * N * D;
        const double* Vh = V + (size_t)h * N * M;
        double* Oh = O + (size_t)h * N * M;
        for (int t = 0; t < N; ++t) {
            for (int e = 0; e < M; ++e) Oh[(size_t)t * M + e] = 0.0;
            double prod = 1.0; /* prod_{l=j+1..t} gamma_l, built as j walks down from t */
            for (int j = t; j >= 0; --j) {
                const double a = prod * dot(Kh + (size_t)j * D, Qh + (size_t)t * D, D);
                for (int e = 0; e < M; ++e) Oh[(size_t)t * M + e] += a * Vh[(size_t)j * M + e];
                prod *= decay_of(h, j, N, H, gamma_head, gates);
            }
        }
    }
}

/* One decode step of the retention recurrence: S = gamma S + k v^T, then
 * out = S^T q.  gamma [nh] (the step's decay of each head), q, k [nh][D],
 * v, out [nh][M]; S [nh][D][M] updated in place. */
void lao_retention_decode_step(int nh, int D, int M, const double* q, const double* k,
                               const double* v, const double* gamma, double* S, double* out) {
    for (int h = 0; h < nh; ++h) {
        double* Sh = S + (size_t)h * D * M;
        for (int d = 0; d < D; ++d)
            for (int e = 0; e < M; ++e)
                Sh[(size_t)d * M + e] = gamma[h] * Sh[(size_t)d * M + e] +
                                        k[(size_t)h * D + d] * v[(size_t)h * M + e];
        for (int e = 0; e < M; ++e) {
            double y = 0.0;
            for (int d = 0; d < D; ++d) y += Sh[(size_t)d * M + e] * q[(size_t)h * D + d];
            out[(size_t)h * M + e] = y;
        }
    }
}

/* ------------------------------------- degree-2 polynomial feature map */

/* "【论文解读】Transformers are RNNs" section 二 (3): the homogeneous
 * polynomial kernel k(x, y) = (x^T y)^2 as the similarity of the general
 * attention form (eq. common), causal (j <= i, eq. mask) or over all j:
 *   V'_i = sum_j (Q_i . K_j)^2 V_j / sum_j (Q_i . K_j)^2
 * written out directly, O(N^2 D) per head. */
void lao_poly_forward_quadratic(int nh, int N, int D, int M, const double* Q, const double* K,
                                const double* V, double* O, int causal) {
    double* num = (double*)malloc(sizeof(double) * (size_t)M);
    for (int h = 0; h < nh; ++h) {
        const double* Qh = Q + (size_t)h * N * D;
        const double* Kh = K + (size_t)h * N * D;
        const double* Vh = V + (size_t)h * N * M;
        double* Oh = O + (size_t)h * N * M;
        for (int i = 0; i < N; ++i) {
            const int jmax = causal ? i : N - 1;
            double den = 0.0;
            memset(num, 0, sizeof(double) * (size_t)M);
            for (int j = 0; j <= jmax; ++j) {
                const double d = dot(Qh + (size_t)i * D, Kh + (size_t)j * D, D);
                const double w = d * d;
                den += w;
                for (int e = 0; e < M; ++e) num[e] += w * Vh[(size_t)j * M + e];
            }
            for (int e = 0; e < M; ++e) Oh[(size_t)i * M + e] = num[e] / den;
        }
    }
    free(num);
}

/* The same through the explicit feature map of that section: phi(x) has the
 * C = D^2 entries x_a x_b (index a D + b), so phi(x) . phi(y) = (x . y)^2, and
 * the linear form keeps S = sum_j phi(K_j) V_j^T (C x M) and Z = sum_j phi(K_j)
 * -- causal: the running sums of section 三 read after each token's update;
 * otherwise the totals.  O(N D^2 M) per head. */
void lao_poly_forward_state(int nh, int N, int D, int M, const double* Q, const double* K,
                            const double* V, double* O, int causal) {
    const int C = D * D;
    double* S = (double*)malloc(sizeof(double) * (size_t)C * M);
    double* Z = (double*)malloc(sizeof(double) * (size_t)C);
    double* f = (double*)malloc(sizeof(double) * (size_t)C);
    for (int h = 0; h < nh; ++h) {
        const double* Qh = Q + (size_t)h * N * D;
        const double* Kh = K + (size_t)h * N * D;
        const double* Vh = V + (size_t)h * N * M;
        double* Oh = O + (size_t)h * N * M;
        memset(S, 0, sizeof(double) * (size_t)C * M);
        memset(Z, 0, sizeof(double) * (size_t)C);
        for (int pass = causal ? 1 : 0; pass < 2; ++pass) {
            /* non-causal: pass 0 forms the totals, pass 1 reads them */
            for (int t = 0; t < N; ++t) {
                if (causal || pass == 0) {
                    const double* k = Kh + (size_t)t * D;
                    for (int a = 0; a < D; ++a)
                        for (int b = 0; b < D; ++b) f[a * D + b] = k[a] * k[b];
                    for (int c = 0; c < C; ++c) {
                        for (int e = 0; e < M; ++e) S[(size_t)c * M + e] += f[c] * Vh[(size_t)t * M + e];
                        Z[c] += f[c];
                    }
                }
                if (pass == 1) {
                    const double* q = Qh + (size_t)t * D;
                    for (int a = 0; a < D; ++a)
                        for (int b = 0; b < D; ++b) f[a * D + b] = q[a] * q[b];
                    const double den = dot(f, Z, C);
                    for (int e = 0; e < M; ++e) {
                        double num = 0.0;
                        for (int c = 0; c < C; ++c) num += f[c] * S[(size_t)c * M + e];
                        Oh[(size_t)t * M + e] = num / den;
                    }
                }
            }
        }
    }
    free(S);
    free(Z);
    free(f);
}
