// retention_ffma.cuh -- linear attention with decay ("retention") on the CUDA
// cores (fp32 FFMA), every dtype and head size.
//
// "Transformer and Variants" (by-xin.github.io) writes linear attention as an
// RNN without the reflection term (section 1.3.2) and adds forgetting in
// section 1.3.4: RetNet H_t = gamma H_{t-1} + v_t k_t^T with one decay gamma,
// gated retention with a decay gamma_t per token, and y_t = H_t q_t.  In the
// S = sum k v^T convention of the rest of the library (S is H transposed):
//     S_t = gamma_t S_{t-1} + k_t v_t^T,   y_t = S_t^T q_t
// with raw q, k (no feature map) and no normaliser; gamma_t = 1 gives the
// plain unnormalised form.
//
// Chunked: inside a chunk of L tokens let a_i be the running sum of
// log2(gamma) over the chunk's tokens 0..i.  Then
//     y_i = sum_{j<=i} 2^(a_i - a_j) (q_i . k_j) v_j + 2^(a_i) q_i^T S_prev
//     S   = 2^(a_{L-1}) S_prev + sum_j 2^(a_{L-1} - a_j) k_j v_j^T
// Every power of two has a non-positive exponent (decays are <= 1).  Spans of
// a head (one CTA each) get their starting state from per-span aggregates
// (decayed to the span's end, with the span's total log2 decay) combined in
// span order.
#pragma once

#include "causal_ffma.cuh"

namespace la {
namespace ffma {

// log2 of a decay, kept finite: a decay below 2^-64 counts as 2^-64 (its
// weight is then below every rounding of the other terms).
__device__ __forceinline__ float log2_decay(float g) { return fmaxf(log2f(g), -64.f); }

// as[i] = sum_{l <= i} log2(gamma_{c0 + l}) for i < L (rows past `rows` keep
// the last value); gates (per token, nullable) else the head's constant lg.
template <int L>
__device__ __forceinline__ void chunk_log_decay(float* as, const float* gates, float lg, int c0,
                                                int rows) {
    if (threadIdx.x == 0) {
        float a = 0.f;
        for (int i = 0; i < L; ++i) {
            if (i < rows) a += gates ? log2_decay(gates[c0 + i]) : lg;
            as[i] = a;
        }
    }
}

__device__ __forceinline__ float head_log_decay(const float* gamma_head, int bh, int H) {
    return gamma_head ? log2_decay(gamma_head[bh % H]) : 0.f;
}

// Per-span aggregate (sum_j 2^(lam - a_j) k_j v_j^T over the span, decayed to
// its end) and the span's total log2 decay lam.
template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
ret_span_aggregate_kernel(const T* __restrict__ K, const T* __restrict__ V,
                          const float* __restrict__ gates, const float* __restrict__ gamma_head,
                          float* __restrict__ agg, float* __restrict__ lam, int N, int H, int spans,
                          int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP;
    extern __shared__ float smem[];
    float* ks = smem;          // [L][DP]
    float* vs = ks + L * DP;   // [L][MP]
    float* as = vs + L * MP;   // [L]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const T* Kh = K + (size_t)bh * N * D;
    const T* Vh = V + (size_t)bh * N * M;
    const float* gh = gates ? gates + (size_t)bh * N : nullptr;
    const float lg = head_log_decay(gamma_head, bh, H);
    Frag<D, M> acc;
    acc.zero();
    float total = 0.f;
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(ks, Kh + (size_t)c0 * D, rows, Ident());
        load_tile<L, M, MP>(vs, Vh + (size_t)c0 * M, rows, Ident());
        chunk_log_decay<L>(as, gh, lg, c0, rows);
        __syncthreads();
        const float A = as[L - 1];
        for (int t = threadIdx.x; t < L * D; t += kThreads) {
            const int j = t / D, d = t - j * D;
            ks[j * DP + d] *= exp2f(A - as[j]);
        }
        __syncthreads();
        const float f = exp2f(A);
        acc.each([&](int, int, float& x) { x *= f; });
        acc.template mac<L>([&](int d, int j) { return ks[j * DP + d]; },
                            [&](int j, int e) { return vs[j * MP + e]; });
        total += A;
    }
    float* out = agg + ((size_t)bh * spans + s) * (D * M);
    acc.each([&](int d, int e, float x) { out[d * M + e] = x; });
    if (threadIdx.x == 0) lam[(size_t)bh * spans + s] = total;
}

// In place: agg[s] becomes the state before span s (S_init decayed plus the
// earlier spans' aggregates, each decayed by the spans after it).
static __global__ void ret_span_scan_kernel(float* __restrict__ agg, const float* __restrict__ lam,
                                            const float* __restrict__ S_init, int BH, int spans,
                                            int DM) {
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)BH * DM) return;
    const int bh = (int)(idx / DM), w = (int)(idx - (size_t)bh * DM);
    float run = S_init ? S_init[idx] : 0.f;
    for (int s = 0; s < spans; ++s) {
        float* p = agg + ((size_t)bh * spans + s) * DM + w;
        const float x = *p;
        *p = run;
        run = exp2f(lam[(size_t)bh * spans + s]) * run + x;
    }
}

template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
ret_forward_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                   T* __restrict__ O, const float* __restrict__ gates,
                   const float* __restrict__ gamma_head, const float* __restrict__ prefix,
                   const float* __restrict__ S_init, float* __restrict__ S_final, int N, int H,
                   int spans, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP, LP = C::LP;
    extern __shared__ float smem[];
    float* Ss = smem;            // [D][MP]
    float* qs = Ss + D * MP;     // [L][DP]
    float* ks = qs + L * DP;     // [L][DP]
    float* vs = ks + L * DP;     // [L][MP]
    float* Ps = vs + L * MP;     // [L][LP]
    float* as = Ps + L * LP;     // [L]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const T* Qh = Q + (size_t)bh * N * D;
    const T* Kh = K + (size_t)bh * N * D;
    const T* Vh = V + (size_t)bh * N * M;
    T* Oh = O + (size_t)bh * N * M;
    const float* gh = gates ? gates + (size_t)bh * N : nullptr;
    const float lg = head_log_decay(gamma_head, bh, H);
    {
        const float* src = prefix ? prefix + ((size_t)bh * spans + s) * (D * M)
                                  : (S_init ? S_init + (size_t)bh * D * M : nullptr);
        for (int t = threadIdx.x; t < D * M; t += kThreads)
            Ss[(t / M) * MP + (t % M)] = src ? src[t] : 0.f;
    }
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(qs, Qh + (size_t)c0 * D, rows, Ident());
        load_tile<L, D, DP>(ks, Kh + (size_t)c0 * D, rows, Ident());
        load_tile<L, M, MP>(vs, Vh + (size_t)c0 * M, rows, Ident());
        chunk_log_decay<L>(as, gh, lg, c0, rows);
        __syncthreads();
        {   // P_ij = 2^(a_i - a_j) (q_i . k_j) for j <= i
            Frag<L, L> p;
            p.zero();
            p.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int j) { return ks[j * DP + d]; });
            p.each([&](int i, int j, float x) {
                Ps[i * LP + j] = j <= i ? x * exp2f(as[i] - as[j]) : 0.f;
            });
        }
        __syncthreads();
        {   // y_i = (P V)_i + 2^(a_i) (q_i^T S_prev)
            Frag<L, M> o, r;
            o.zero();
            r.zero();
            o.template mac<L>([&](int i, int j) { return Ps[i * LP + j]; },
                              [&](int j, int e) { return vs[j * MP + e]; });
            r.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int e) { return Ss[d * MP + e]; });
            const int ty = threadIdx.x >> 4;  // this thread's rows are ty + 16 a
#pragma unroll
            for (int a = 0; a < Frag<L, M>::TR; ++a) {
                const float f = exp2f(as[ty + 16 * a]);
#pragma unroll
                for (int b = 0; b < Frag<L, M>::TC; ++b) o.v[a][b] = fmaf(f, r.v[a][b], o.v[a][b]);
            }
            o.each([&](int i, int e, float x) {
                if (i < rows) Oh[(size_t)(c0 + i) * M + e] = from_f<T>(x);
            });
        }
        __syncthreads();
        {   // S = 2^A S_prev + sum_j 2^(A - a_j) k_j v_j^T
            const float A = as[L - 1];
            for (int t = threadIdx.x; t < L * D; t += kThreads) {
                const int j = t / D, d = t - j * D;
                ks[j * DP + d] *= exp2f(A - as[j]);
            }
            __syncthreads();
            Frag<D, M> u;
            u.zero();
            u.template mac<L>([&](int d, int j) { return ks[j * DP + d]; },
                              [&](int j, int e) { return vs[j * MP + e]; });
            const float f = exp2f(A);
            u.each([&](int d, int e, float x) { Ss[d * MP + e] = f * Ss[d * MP + e] + x; });
        }
    }
    if (S_final && s == spans - 1) {
        __syncthreads();
        for (int t = threadIdx.x; t < D * M; t += kThreads)
            S_final[(size_t)bh * D * M + t] = Ss[(t / M) * MP + (t % M)];
    }
}

template <int D, int M>
struct RetSmem {
    using C = Cfg<D, M>;
    static constexpr size_t agg = sizeof(float) * (C::L * C::DP + C::L * C::MP + C::L);
    static constexpr size_t fwd =
        sizeof(float) * (D * C::MP + 2 * C::L * C::DP + C::L * C::MP + C::L * C::LP + C::L);
};

}  // namespace ffma

template <typename T, int D, int M>
cudaError_t retention_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O,
                              const float* gamma_head, const float* gates, int BH, int H, int N,
                              const float* S_init, float* S_final) {
    using namespace ffma;
    using C = Cfg<D, M>;
    int spans, span_len;
    choose_spans(BH, N, C::L, c.num_sms, &spans, &span_len);
    float* agg = nullptr;
    float* lam = nullptr;
    if (spans > 1) {
        LA_TRY(scratch_alloc(c, (void**)&agg, plan::ffma_retention_forward(BH, N, D, M, c.num_sms)));
        lam = agg + (size_t)BH * spans * D * M;
        LA_TRY(allow_smem(ret_span_aggregate_kernel<T, D, M>, RetSmem<D, M>::agg));
        ret_span_aggregate_kernel<T, D, M><<<dim3(BH, spans), kThreads, RetSmem<D, M>::agg, c.stream>>>(
            K, V, gates, gamma_head, agg, lam, N, H, spans, span_len);
        const size_t n = (size_t)BH * D * M;
        ret_span_scan_kernel<<<(unsigned)((n + 255) / 256), 256, 0, c.stream>>>(agg, lam, S_init, BH,
                                                                                spans, D * M);
        note_launch(2);
    }
    LA_TRY(allow_smem(ret_forward_kernel<T, D, M>, RetSmem<D, M>::fwd));
    ret_forward_kernel<T, D, M><<<dim3(BH, spans), kThreads, RetSmem<D, M>::fwd, c.stream>>>(
        Q, K, V, O, gates, gamma_head, agg, S_init, S_final, N, H, spans, span_len);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (agg) scratch_free(c, agg);
    return e;
}

}  // namespace la
