// causal_ffma.cuh -- chunked causal linear attention on the CUDA cores (fp32 FFMA).
//
// A head's sequence is cut into spans (one CTA each) and each span into chunks
// of L tokens.  Inside a chunk c of a span the causal sums split into
//   intra-chunk:  P = tril(phi(Q_c) phi(K_c)^T) (diagonal kept),  P V_c,  rowsum(P)
//   inter-chunk:  phi(Q_c) S_{c-1},  phi(Q_c) Z_{c-1}
// and the state moves on by S_c = S_{c-1} + phi(K_c)^T V_c, Z_c = Z_{c-1} +
// colsum phi(K_c) -- the incremental update of "Transformers are RNNs"
// section 三 applied a chunk at a time.  Spans get their starting state from
// an exclusive scan over per-span aggregates (a separate pass over K, V).
//
// The backward follows section 三（一）4 (eqs. gq-gv): a prefix pass for
// dphi(Q) with the state S, Z, then a suffix pass over chunks in reverse for
// dphi(K) and dV with R = sum_{j>=i} phi(Q_j) gn_j^T, r = sum_{j>=i} phi(Q_j) gd_j,
// where gn = G / den and gd = -(G . O) / den carry the quotient rule.
#pragma once

#include <algorithm>

#include "la_common.cuh"
#include "la_launch.h"
#include "la_plan.h"

namespace la {
namespace ffma {

constexpr int kThreads = 256;

template <int D, int M>
struct Cfg {
    static constexpr int L = plan::ffma_chunk(D, M);                 // chunk length
    static constexpr int W = static_cast<int>(plan::state_words(D, M));  // state words (S | Z)
    static constexpr int DP = D + 1;                               // padded row strides
    static constexpr int MP = M + 1;
    static constexpr int LP = L + 1;
};

// Loads `rows` valid rows of a [*, C] tile starting at row n0 into smem with
// row stride CP, applying `f` to each value; rows >= `rows` are zero.
template <int R, int C, int CP, typename T, class F>
__device__ __forceinline__ void load_tile(float* dst, const T* __restrict__ src, int rows, F f) {
    for (int t = threadIdx.x; t < R * C; t += kThreads) {
        const int r = t / C, c = t - (t / C) * C;
        dst[r * CP + c] = r < rows ? f(to_f(src[(size_t)r * C + c])) : 0.f;
    }
}

struct Ident {
    __device__ __forceinline__ float operator()(float x) const { return x; }
};
struct Phi {
    __device__ __forceinline__ float operator()(float x) const { return phi(x); }
};

// --------------------------------------------------------------------------
// Per-span aggregates A_s = (sum_{j in span} phi(K_j) V_j^T | sum phi(K_j)).
template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
span_aggregate_kernel(const T* __restrict__ K, const T* __restrict__ V, float* __restrict__ agg,
                      int N, int spans, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L;
    extern __shared__ float smem[];
    float* ks = smem;
    float* vs = ks + L * C::DP;
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const T* Kh = K + (size_t)bh * N * D;
    const T* Vh = V + (size_t)bh * N * M;
    Frag<D, M> acc;
    acc.zero();
    float z = 0.f;  // thread d < D owns Z[d]
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, C::DP>(ks, Kh + (size_t)c0 * D, rows, Phi());
        load_tile<L, M, C::MP>(vs, Vh + (size_t)c0 * M, rows, Ident());
        __syncthreads();
        acc.template mac<L>([&](int d, int j) { return ks[j * C::DP + d]; },
                            [&](int j, int e) { return vs[j * C::MP + e]; });
        if (threadIdx.x < D)
            for (int j = 0; j < L; ++j) z += ks[j * C::DP + threadIdx.x];
    }
    float* out = agg + ((size_t)bh * spans + s) * C::W;
    acc.each([&](int d, int e, float x) { out[d * M + e] = x; });
    if (threadIdx.x < D) out[D * M + threadIdx.x] = z;
}

// Exclusive scan of span aggregates in place, in span order or (reverse) in
// reverse span order, starting from an optional initial state; the running
// total after the last span goes to `totals` when given.
static __global__ void span_scan_kernel(float* __restrict__ agg, const float* __restrict__ S_init,
                                 const float* __restrict__ Z_init, float* __restrict__ totals,
                                 int BH, int spans, int D, int M, int reverse) {
    const int W = D * M + D;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)BH * W) return;
    const int bh = (int)(idx / W), w = (int)(idx - (size_t)bh * W);
    float run = 0.f;
    if (S_init) run = w < D * M ? S_init[(size_t)bh * D * M + w] : Z_init[(size_t)bh * D + (w - D * M)];
    for (int t = 0; t < spans; ++t) {
        const int s = reverse ? spans - 1 - t : t;
        float* p = agg + ((size_t)bh * spans + s) * W + w;
        const float x = *p;
        *p = run;
        run += x;
    }
    if (totals) totals[idx] = run;
}

// Loads a (S | Z) state word vector into padded smem S [D][M+1] and Z [D].
template <int D, int M>
__device__ __forceinline__ void load_state(float* Ss, float* Zs, const float* src,
                                           const float* S_init, const float* Z_init) {
    for (int t = threadIdx.x; t < D * M + D; t += kThreads) {
        float x = 0.f;
        if (src) x = src[t];
        else if (S_init) x = t < D * M ? S_init[t] : Z_init[t - D * M];
        if (t < D * M) Ss[(t / M) * (M + 1) + (t % M)] = x;
        else Zs[t - D * M] = x;
    }
}

// den_i = sum_j P_ij + phi(Q_i) . Z  (one warp per row).
template <int D, int L>
__device__ __forceinline__ void row_den(float* dens, const float* Ps, const float* qs,
                                        const float* Zs) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < L; i += kThreads / 32) {
        float a = 0.f;
        for (int j = lane; j < L; j += 32) a += Ps[i * (L + 1) + j];
        for (int d = lane; d < D; d += 32) a = fmaf(qs[i * (D + 1) + d], Zs[d], a);
#pragma unroll
        for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) dens[i] = a;
    }
}

// --------------------------------------------------------------------------
// Forward over one span.
template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
causal_forward_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                      T* __restrict__ O, const float* __restrict__ prefix,
                      const float* __restrict__ S_init, const float* __restrict__ Z_init,
                      float* __restrict__ S_final, float* __restrict__ Z_final,
                      float* __restrict__ Den, int N, int spans, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP, LP = C::LP;
    extern __shared__ float smem[];
    float* Ss = smem;            // [D][MP]
    float* Zs = Ss + D * MP;     // [D]
    float* qs = Zs + D;          // [L][DP]
    float* ks = qs + L * DP;     // [L][DP]
    float* vs = ks + L * DP;     // [L][MP]
    float* Ps = vs + L * MP;     // [L][LP]
    float* dens = Ps + L * LP;   // [L]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const T* Qh = Q + (size_t)bh * N * D;
    const T* Kh = K + (size_t)bh * N * D;
    const T* Vh = V + (size_t)bh * N * M;
    T* Oh = O + (size_t)bh * N * M;

    load_state<D, M>(Ss, Zs, prefix ? prefix + ((size_t)bh * spans + s) * C::W : nullptr,
                     S_init ? S_init + (size_t)bh * D * M : nullptr,
                     Z_init ? Z_init + (size_t)bh * D : nullptr);
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(qs, Qh + (size_t)c0 * D, rows, Phi());
        load_tile<L, D, DP>(ks, Kh + (size_t)c0 * D, rows, Phi());
        load_tile<L, M, MP>(vs, Vh + (size_t)c0 * M, rows, Ident());
        __syncthreads();
        {   // P = tril(phi(Q_c) phi(K_c)^T)
            Frag<L, L> p;
            p.zero();
            p.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int j) { return ks[j * DP + d]; });
            p.each([&](int i, int j, float x) { Ps[i * LP + j] = j <= i ? x : 0.f; });
        }
        __syncthreads();
        row_den<D, L>(dens, Ps, qs, Zs);
        __syncthreads();
        if (Den)  // the normaliser, kept for the backward
            for (int i = threadIdx.x; i < rows; i += kThreads) Den[(size_t)bh * N + c0 + i] = dens[i];
        {   // O_c = (P V_c + phi(Q_c) S_{c-1}) / den
            Frag<L, M> o;
            o.zero();
            o.template mac<L>([&](int i, int j) { return Ps[i * LP + j]; },
                              [&](int j, int e) { return vs[j * MP + e]; });
            o.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int e) { return Ss[d * MP + e]; });
            o.each([&](int i, int e, float x) {
                if (i < rows) Oh[(size_t)(c0 + i) * M + e] = from_f<T>(x / dens[i]);
            });
        }
        __syncthreads();
        {   // S += phi(K_c)^T V_c, Z += colsum phi(K_c)
            Frag<D, M> u;
            u.zero();
            u.template mac<L>([&](int d, int j) { return ks[j * DP + d]; },
                              [&](int j, int e) { return vs[j * MP + e]; });
            u.each([&](int d, int e, float x) { Ss[d * MP + e] += x; });
            if (threadIdx.x < D) {
                float z = 0.f;
                for (int j = 0; j < L; ++j) z += ks[j * DP + threadIdx.x];
                Zs[threadIdx.x] += z;
            }
        }
    }
    if (S_final && s == spans - 1) {
        __syncthreads();
        for (int t = threadIdx.x; t < D * M; t += kThreads)
            S_final[(size_t)bh * D * M + t] = Ss[(t / M) * MP + (t % M)];
        for (int t = threadIdx.x; t < D; t += kThreads) Z_final[(size_t)bh * D + t] = Zs[t];
    }
}

// --------------------------------------------------------------------------
// Backward, prefix direction: den, (O), gn, gd, dQ; per-span (sum phi(Q) gn^T | sum phi(Q) gd).
template <typename T, int D, int M, bool HAS_O>
__global__ void __launch_bounds__(kThreads)
backward_prefix_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                       const T* __restrict__ Oin, const T* __restrict__ G, T* __restrict__ dQ,
                       float* __restrict__ gn_ws, float* __restrict__ gd_ws,
                       const float* __restrict__ prefix, float* __restrict__ ragg, int N,
                       int spans, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP, LP = C::LP;
    extern __shared__ float smem[];
    float* Ss = smem;            // [D][MP]
    float* Zs = Ss + D * MP;     // [D]
    float* rsum = Zs + D;        // [D]  sum_i phi(Q_i) gd_i over the span
    float* qs = rsum + D;        // [L][DP]
    float* ks = qs + L * DP;     // [L][DP]
    float* vs = ks + L * DP;     // [L][MP]
    float* gs = vs + L * MP;     // [L][MP]  G, then gn
    float* os = gs + L * MP;     // [L][MP]
    float* Ps = os + L * MP;     // [L][LP]  P, then dP
    float* dens = Ps + L * LP;   // [L]
    float* gds = dens + L;       // [L]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const size_t hq = (size_t)bh * N * D, hv = (size_t)bh * N * M;

    load_state<D, M>(Ss, Zs, prefix ? prefix + ((size_t)bh * spans + s) * C::W : nullptr,
                     nullptr, nullptr);
    for (int t = threadIdx.x; t < D; t += kThreads) rsum[t] = 0.f;
    Frag<D, M> racc;
    racc.zero();
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(qs, Q + hq + (size_t)c0 * D, rows, Phi());
        load_tile<L, D, DP>(ks, K + hq + (size_t)c0 * D, rows, Phi());
        load_tile<L, M, MP>(vs, V + hv + (size_t)c0 * M, rows, Ident());
        load_tile<L, M, MP>(gs, G + hv + (size_t)c0 * M, rows, Ident());
        if (HAS_O) load_tile<L, M, MP>(os, Oin + hv + (size_t)c0 * M, rows, Ident());
        __syncthreads();
        {
            Frag<L, L> p;
            p.zero();
            p.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int j) { return ks[j * DP + d]; });
            p.each([&](int i, int j, float x) { Ps[i * LP + j] = j <= i ? x : 0.f; });
        }
        __syncthreads();
        row_den<D, L>(dens, Ps, qs, Zs);
        __syncthreads();
        if (!HAS_O) {
            Frag<L, M> o;
            o.zero();
            o.template mac<L>([&](int i, int j) { return Ps[i * LP + j]; },
                              [&](int j, int e) { return vs[j * MP + e]; });
            o.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int e) { return Ss[d * MP + e]; });
            o.each([&](int i, int e, float x) { os[i * MP + e] = i < rows ? x / dens[i] : 0.f; });
            __syncthreads();
        }
        {   // gd_i = -(G_i . O_i) / den_i   (zero for padding rows)
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            for (int i = warp; i < L; i += kThreads / 32) {
                float a = 0.f;
                for (int e = lane; e < M; e += 32) a = fmaf(gs[i * MP + e], os[i * MP + e], a);
#pragma unroll
                for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                if (lane == 0) gds[i] = i < rows ? -a / dens[i] : 0.f;
            }
        }
        __syncthreads();
        for (int t = threadIdx.x; t < L * M; t += kThreads) {  // gn = G / den
            const int i = t / M, e = t - (t / M) * M;
            const float g = i < rows ? gs[i * MP + e] / dens[i] : 0.f;
            gs[i * MP + e] = g;
            if (i < rows) gn_ws[hv + (size_t)(c0 + i) * M + e] = g;
        }
        for (int i = threadIdx.x; i < rows; i += kThreads) gd_ws[(size_t)bh * N + c0 + i] = gds[i];
        __syncthreads();
        {   // dP = tril(gn V^T + gd 1^T)
            Frag<L, L> p;
            p.zero();
            p.template mac<M>([&](int i, int e) { return gs[i * MP + e]; },
                              [&](int e, int j) { return vs[j * MP + e]; });
            p.each([&](int i, int j, float x) { Ps[i * LP + j] = j <= i ? x + gds[i] : 0.f; });
        }
        __syncthreads();
        {   // dphi(Q) = dP phi(K) + gn S^T + gd Z^T;  dQ = dphi(Q) * phi'(Q)
            Frag<L, D> q;
            q.zero();
            q.template mac<L>([&](int i, int j) { return Ps[i * LP + j]; },
                              [&](int j, int d) { return ks[j * DP + d]; });
            q.template mac<M>([&](int i, int e) { return gs[i * MP + e]; },
                              [&](int e, int d) { return Ss[d * MP + e]; });
            q.each([&](int i, int d, float x) {
                if (i < rows) {
                    x = fmaf(gds[i], Zs[d], x);
                    dQ[hq + (size_t)(c0 + i) * D + d] = from_f<T>(x * dphi_from_phi(qs[i * DP + d]));
                }
            });
        }
        // span sums of phi(Q) gn^T and phi(Q) gd (for the suffix pass)
        racc.template mac<L>([&](int d, int i) { return qs[i * DP + d]; },
                             [&](int i, int e) { return gs[i * MP + e]; });
        if (threadIdx.x < D) {
            float a = 0.f;
            for (int i = 0; i < L; ++i) a = fmaf(qs[i * DP + threadIdx.x], gds[i], a);
            rsum[threadIdx.x] += a;
        }
        __syncthreads();
        {   // S += phi(K_c)^T V_c, Z += colsum phi(K_c)
            Frag<D, M> u;
            u.zero();
            u.template mac<L>([&](int d, int j) { return ks[j * DP + d]; },
                              [&](int j, int e) { return vs[j * MP + e]; });
            u.each([&](int d, int e, float x) { Ss[d * MP + e] += x; });
            if (threadIdx.x < D) {
                float z = 0.f;
                for (int j = 0; j < L; ++j) z += ks[j * DP + threadIdx.x];
                Zs[threadIdx.x] += z;
            }
        }
    }
    __syncthreads();
    float* out = ragg + ((size_t)bh * spans + s) * C::W;
    racc.each([&](int d, int e, float x) { out[d * M + e] = x; });
    for (int t = threadIdx.x; t < D; t += kThreads) out[D * M + t] = rsum[t];
}

// Backward, suffix direction over chunks in reverse: dK, dV.
template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
backward_suffix_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                       const float* __restrict__ gn_ws, const float* __restrict__ gd_ws,
                       T* __restrict__ dK, T* __restrict__ dV, const float* __restrict__ suffix,
                       int N, int spans, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP, LP = C::LP;
    extern __shared__ float smem[];
    float* Rs = smem;            // [D][MP]  R = sum_{later} phi(Q) gn^T
    float* rs = Rs + D * MP;     // [D]      r = sum_{later} phi(Q) gd
    float* qs = rs + D;          // [L][DP]
    float* ks = qs + L * DP;     // [L][DP]
    float* vs = ks + L * DP;     // [L][MP]
    float* gns = vs + L * MP;    // [L][MP]
    float* Ps = gns + L * MP;    // [L][LP]
    float* dPs = Ps + L * LP;    // [L][LP]
    float* gds = dPs + L * LP;   // [L]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const size_t hq = (size_t)bh * N * D, hv = (size_t)bh * N * M;
    load_state<D, M>(Rs, rs, suffix ? suffix + ((size_t)bh * spans + s) * C::W : nullptr,
                     nullptr, nullptr);
    const int nchunks = (n1 - n0 + L - 1) / L;
    for (int c = nchunks - 1; c >= 0; --c) {
        const int c0 = n0 + c * L;
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(qs, Q + hq + (size_t)c0 * D, rows, Phi());
        load_tile<L, D, DP>(ks, K + hq + (size_t)c0 * D, rows, Phi());
        load_tile<L, M, MP>(vs, V + hv + (size_t)c0 * M, rows, Ident());
        for (int t = threadIdx.x; t < L * M; t += kThreads) {
            const int i = t / M, e = t - (t / M) * M;
            gns[i * MP + e] = i < rows ? gn_ws[hv + (size_t)(c0 + i) * M + e] : 0.f;
        }
        for (int i = threadIdx.x; i < L; i += kThreads)
            gds[i] = i < rows ? gd_ws[(size_t)bh * N + c0 + i] : 0.f;
        __syncthreads();
        {
            Frag<L, L> p;
            p.zero();
            p.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int j) { return ks[j * DP + d]; });
            p.each([&](int i, int j, float x) { Ps[i * LP + j] = j <= i ? x : 0.f; });
            Frag<L, L> g;
            g.zero();
            g.template mac<M>([&](int i, int e) { return gns[i * MP + e]; },
                              [&](int e, int j) { return vs[j * MP + e]; });
            g.each([&](int i, int j, float x) { dPs[i * LP + j] = j <= i ? x + gds[i] : 0.f; });
        }
        __syncthreads();
        {   // dphi(K_j) = sum_{i>=j} dP_ij phi(Q_i) + R V_j + r;  dK = dphi(K) * phi'(K)
            Frag<L, D> k;
            k.zero();
            k.template mac<L>([&](int j, int i) { return dPs[i * LP + j]; },
                              [&](int i, int d) { return qs[i * DP + d]; });
            k.template mac<M>([&](int j, int e) { return vs[j * MP + e]; },
                              [&](int e, int d) { return Rs[d * MP + e]; });
            k.each([&](int j, int d, float x) {
                if (j < rows)
                    dK[hq + (size_t)(c0 + j) * D + d] =
                        from_f<T>((x + rs[d]) * dphi_from_phi(ks[j * DP + d]));
            });
            // dV_j = sum_{i>=j} P_ij gn_i + R^T phi(K_j)
            Frag<L, M> v;
            v.zero();
            v.template mac<L>([&](int j, int i) { return Ps[i * LP + j]; },
                              [&](int i, int e) { return gns[i * MP + e]; });
            v.template mac<D>([&](int j, int d) { return ks[j * DP + d]; },
                              [&](int d, int e) { return Rs[d * MP + e]; });
            v.each([&](int j, int e, float x) {
                if (j < rows) dV[hv + (size_t)(c0 + j) * M + e] = from_f<T>(x);
            });
        }
        __syncthreads();
        {   // R += phi(Q_c)^T gn_c, r += phi(Q_c)^T gd_c
            Frag<D, M> u;
            u.zero();
            u.template mac<L>([&](int d, int i) { return qs[i * DP + d]; },
                              [&](int i, int e) { return gns[i * MP + e]; });
            u.each([&](int d, int e, float x) { Rs[d * MP + e] += x; });
            if (threadIdx.x < D) {
                float a = 0.f;
                for (int i = 0; i < L; ++i) a = fmaf(qs[i * DP + threadIdx.x], gds[i], a);
                rs[threadIdx.x] += a;
            }
        }
    }
}

// --------------------------------------------------------------------------
// Host side.

template <int D, int M>
struct Smem {
    using C = Cfg<D, M>;
    static constexpr size_t agg = sizeof(float) * (C::L * C::DP + C::L * C::MP);
    static constexpr size_t fwd =
        sizeof(float) * (D * C::MP + D + 2 * C::L * C::DP + C::L * C::MP + C::L * C::LP + C::L);
    static constexpr size_t bwd_prefix = sizeof(float) * (D * C::MP + 2 * D + 2 * C::L * C::DP +
                                                          3 * C::L * C::MP + C::L * C::LP + 2 * C::L);
    static constexpr size_t bwd_suffix = sizeof(float) * (D * C::MP + D + 2 * C::L * C::DP +
                                                          2 * C::L * C::MP + 2 * C::L * C::LP + C::L);
};

// Spans per head: enough CTAs for about two per SM, whole chunks per span.
inline void choose_spans(int BH, int N, int L, int num_sms, int* spans, int* span_len) {
    plan::ffma_spans(BH, N, L, num_sms, spans, span_len);
}

template <class K>
inline cudaError_t allow_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace ffma

#define LA_TRY(expr)                         \
    do {                                     \
        cudaError_t _e = (expr);             \
        if (_e != cudaSuccess) return _e;    \
    } while (0)

template <typename T, int D, int M>
cudaError_t causal_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O, int BH,
                           int N, const float* S_init, const float* Z_init, float* S_final,
                           float* Z_final, float* Den) {
    using namespace ffma;
    using C = Cfg<D, M>;
    int spans, span_len;
    choose_spans(BH, N, C::L, c.num_sms, &spans, &span_len);
    float* agg = nullptr;
    if (spans > 1) {
        LA_TRY(scratch_alloc(c, (void**)&agg, plan::ffma_causal_forward(BH, N, D, M, c.num_sms)));
        LA_TRY(allow_smem(span_aggregate_kernel<T, D, M>, Smem<D, M>::agg));
        span_aggregate_kernel<T, D, M><<<dim3(BH, spans), kThreads, Smem<D, M>::agg, c.stream>>>(
            K, V, agg, N, spans, span_len);
        const size_t n = (size_t)BH * C::W;
        span_scan_kernel<<<(unsigned)((n + 255) / 256), 256, 0, c.stream>>>(
            agg, S_init, Z_init, nullptr, BH, spans, D, M, 0);
        note_launch(2);
    }
    LA_TRY(allow_smem(causal_forward_kernel<T, D, M>, Smem<D, M>::fwd));
    causal_forward_kernel<T, D, M><<<dim3(BH, spans), kThreads, Smem<D, M>::fwd, c.stream>>>(
        Q, K, V, O, agg, S_init, Z_init, S_final, Z_final, Den, N, spans, span_len);
    note_launch();
    cudaError_t e = cudaGetLastError();
    if (agg) scratch_free(c, agg);
    return e;
}

template <typename T, int D, int M>
cudaError_t causal_backward(const LaunchCtx& c, const T* Q, const T* K, const T* V, const T* O,
                            const T* G, T* dQ, T* dK, T* dV, int BH, int N) {
    using namespace ffma;
    using C = Cfg<D, M>;
    int spans, span_len;
    choose_spans(BH, N, C::L, c.num_sms, &spans, &span_len);
    const size_t agg_bytes = sizeof(float) * (size_t)BH * spans * C::W;
    const size_t gn_bytes = sizeof(float) * (size_t)BH * N * M;
    char* ws = nullptr;
    LA_TRY(scratch_alloc(c, (void**)&ws, plan::ffma_causal_backward(BH, N, D, M, c.num_sms)));
    float* sagg = (float*)ws;
    float* ragg = (float*)(ws + agg_bytes);
    float* gn = (float*)(ws + 2 * agg_bytes);
    float* gd = (float*)(ws + 2 * agg_bytes + gn_bytes);
    const size_t n = (size_t)BH * C::W;
    const unsigned scan_grid = (unsigned)((n + 255) / 256);
    cudaError_t e = cudaSuccess;
    do {
        if (spans > 1) {
            if ((e = allow_smem(span_aggregate_kernel<T, D, M>, Smem<D, M>::agg))) break;
            span_aggregate_kernel<T, D, M><<<dim3(BH, spans), kThreads, Smem<D, M>::agg, c.stream>>>(
                K, V, sagg, N, spans, span_len);
            span_scan_kernel<<<scan_grid, 256, 0, c.stream>>>(sagg, nullptr, nullptr, nullptr, BH,
                                                              spans, D, M, 0);
            note_launch(2);
        }
        if (O) {
            if ((e = allow_smem(backward_prefix_kernel<T, D, M, true>, Smem<D, M>::bwd_prefix))) break;
            backward_prefix_kernel<T, D, M, true>
                <<<dim3(BH, spans), kThreads, Smem<D, M>::bwd_prefix, c.stream>>>(
                    Q, K, V, O, G, dQ, gn, gd, spans > 1 ? sagg : nullptr, ragg, N, spans, span_len);
        } else {
            if ((e = allow_smem(backward_prefix_kernel<T, D, M, false>, Smem<D, M>::bwd_prefix))) break;
            backward_prefix_kernel<T, D, M, false>
                <<<dim3(BH, spans), kThreads, Smem<D, M>::bwd_prefix, c.stream>>>(
                    Q, K, V, O, G, dQ, gn, gd, spans > 1 ? sagg : nullptr, ragg, N, spans, span_len);
        }
        note_launch();
        if (spans > 1) {
            span_scan_kernel<<<scan_grid, 256, 0, c.stream>>>(ragg, nullptr, nullptr, nullptr, BH,
                                                              spans, D, M, 1);
            note_launch();
        }
        if ((e = allow_smem(backward_suffix_kernel<T, D, M>, Smem<D, M>::bwd_suffix))) break;
        backward_suffix_kernel<T, D, M>
            <<<dim3(BH, spans), kThreads, Smem<D, M>::bwd_suffix, c.stream>>>(
                Q, K, V, gn, gd, dK, dV, spans > 1 ? ragg : nullptr, N, spans, span_len);
        note_launch();
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, ws);
    return e;
}

}  // namespace la
