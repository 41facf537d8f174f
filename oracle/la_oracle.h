/*
 * la_oracle.h -- plain fp64 CPU oracle for kernelized linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this code: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no header, helper or table with the CUDA
 * library.
 *
 * Source: "【论文解读】Transformers are RNNs" (wkq9411.github.io), sections
 * 二 (eq. common, eq. linear), 特征映射 (eq. elu), 三 (eq. mask, the S/Z
 * definitions, the incremental update, eq. output), 三（一） (numerator
 * gradients, eqs. gq-gv) and 四 (the RNN form); decode order from
 * "Transformer与RNN的深层联结" (xxqk.cn) section 2, RNN-mode inference.
 *
 * Layout: every tensor is a contiguous row-major double array over nh = B*H
 * independent heads: Q, K [nh][N][D]; V, O, G [nh][N][M]; S [nh][D][M];
 * Z [nh][D].  No scaling of Q or K is applied (the pages apply phi to the raw
 * projections).  The causal mask keeps j <= i (diagonal included).
 */
#ifndef LA_ORACLE_H
#define LA_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/* phi(x) = elu(x) + 1 with alpha = 1, and its derivative. */
double lao_phi(double x);
double lao_dphi(double x);

/* Number of host threads the threaded routines use when nthreads <= 0. */
int lao_default_threads(void);

/* Causal forward, quadratic form: O_i = sum_{j<=i} w_ij V_j / sum_{j<=i} w_ij,
 * w_ij = phi(Q_i).phi(K_j).  O(N^2) per head. */
void lao_causal_forward_quadratic(int nh, int N, int D, int M, const double* Q,
                                  const double* K, const double* V, double* O);

/* Causal forward, recurrent S/Z form.  S0/Z0 (nullable) give the state before
 * the first token; S_out/Z_out (nullable) receive the state after the last;
 * den_out (nullable, [nh][N]) the denominator phi(Q_t)^T Z_t of every token. */
void lao_causal_forward_recurrent(int nh, int N, int D, int M, const double* Q,
                                  const double* K, const double* V,
                                  const double* S0, const double* Z0, double* O,
                                  double* S_out, double* Z_out, double* den_out, int nthreads);

/* Non-causal forward, quadratic form (sums over all j). */
void lao_noncausal_forward_quadratic(int nh, int N, int D, int M, const double* Q,
                                     const double* K, const double* V, double* O);

/* Non-causal forward, associativity form phi(Q)(phi(K)^T V) / phi(Q).sum phi(K).
 * S_out/Z_out (nullable) receive S = phi(K)^T V and Z = sum_j phi(K_j). */
void lao_noncausal_forward_assoc(int nh, int N, int D, int M, const double* Q,
                                 const double* K, const double* V, double* O,
                                 double* S_out, double* Z_out, int nthreads);

/* Causal backward, cumulative-sum form: prefix state for dphi(Q), suffix state
 * for dphi(K) and dV; the denominator by the quotient rule. */
void lao_causal_backward_cumsum(int nh, int N, int D, int M, const double* Q,
                                const double* K, const double* V, const double* G,
                                double* dQ, double* dK, double* dV, int nthreads);

/* Causal backward, quadratic form (derivative of the masked quotient). */
void lao_causal_backward_quadratic(int nh, int N, int D, int M, const double* Q,
                                   const double* K, const double* V, const double* G,
                                   double* dQ, double* dK, double* dV);

/* Non-causal backward, state form: the gradients of section 三（一）4 with
 * the prefix and suffix states taken over all tokens (S, Z and R, r are
 * totals), the denominator by the quotient rule. */
void lao_noncausal_backward_assoc(int nh, int N, int D, int M, const double* Q,
                                  const double* K, const double* V, const double* G,
                                  double* dQ, double* dK, double* dV, int nthreads);

/* Non-causal backward, quadratic form (derivative of the unmasked quotient). */
void lao_noncausal_backward_quadratic(int nh, int N, int D, int M, const double* Q,
                                      const double* K, const double* V, const double* G,
                                      double* dQ, double* dK, double* dV);

/* One recurrent decode step for nh heads: S += phi(k) v^T, Z += phi(k), then
 * out = phi(q)^T S / phi(q).Z (update first, then read).  q,k [nh][D],
 * v, out [nh][M]; S, Z updated in place. */
void lao_decode_step(int nh, int D, int M, const double* q, const double* k,
                     const double* v, double* S, double* Z, double* out);

/* Softmax attention decode step with a KV cache: append (k, v) to the T
 * cached positions, then out = softmax(q K^T / sqrt(D)) V over all T + 1.
 * q, k [nh][D]; v, out [nh][M]; Kc [nh][T][D], Vc [nh][T][M] (read only). */
void lao_softmax_decode_step(int nh, int T, int D, int M, const double* q, const double* k,
                             const double* v, const double* Kc, const double* Vc, double* out);

/* Retention ("Transformer and Variants" sections 1.3.2 and 1.3.4): S_t =
 * gamma_t S_{t-1} + k_t v_t^T, y_t = S_t^T q_t, raw q, k, no normaliser.
 * gamma_t = gates[h][t] if gates, else gamma_head[h % H] if gamma_head, else 1
 * (h over nh = B*H heads).  Recurrent form (with optional S0 / S_out) and the
 * unrolled sum over j <= t. */
void lao_retention_forward_recurrent(int nh, int H, int N, int D, int M, const double* Q,
                                     const double* K, const double* V, const double* gamma_head,
                                     const double* gates, const double* S0, double* O,
                                     double* S_out);
void lao_retention_forward_quadratic(int nh, int H, int N, int D, int M, const double* Q,
                                     const double* K, const double* V, const double* gamma_head,
                                     const double* gates, double* O);
/* One retention decode step per head: S = gamma S + k v^T, out = S^T q. */
void lao_retention_decode_step(int nh, int D, int M, const double* q, const double* k,
                               const double* v, const double* gamma, double* S, double* out);

/* Degree-2 polynomial similarity (x^T y)^2 ("Transformers are RNNs" section
 * 二 (3)): the quadratic form, and the linear form through the explicit
 * feature map phi(x) = (x_a x_b), C = D^2 (state S: C x M, Z: C).  causal != 0
 * keeps j <= i. */
void lao_poly_forward_quadratic(int nh, int N, int D, int M, const double* Q, const double* K,
                                const double* V, double* O, int causal);
void lao_poly_forward_state(int nh, int N, int D, int M, const double* Q, const double* K,
                            const double* V, double* O, int causal);

#ifdef __cplusplus
}
#endif
#endif
