// noncausal_bwd_ffma.cuh -- backward of non-causal linear attention on the
// CUDA cores (fp32 FFMA), every dtype and head size.
//
// With O = phi(Q) S / phi(Q) Z, S = phi(K)^T V, Z = sum_j phi(K_j) ("Transformers
// are RNNs", section 二, eq. linear), the gradients of section 三（一）4
// (eqs. gq-gv) take their prefix and suffix sums over every token, and the
// denominator enters by the quotient rule:
//   gn_i = G_i / den_i,  gd_i = -(G_i . O_i) / den_i
//   dphi(Q_i) = S gn_i + Z gd_i
//   R = sum_i phi(Q_i) gn_i^T,  r = sum_i phi(Q_i) gd_i
//   dphi(K_j) = R V_j + r,  dV_j = R^T phi(K_j)
// and dQ, dK by the chain rule through phi.  Three passes, each over spans of
// a head (one CTA per (head, span)): the state (S | Z) as per-span partials
// reduced in span order; the query side (dQ and per-span partials of (R | r));
// the key side (dK, dV).
#pragma once

#include "noncausal_ffma.cuh"

namespace la {
namespace ffma {

// Query side over one span: dQ and this span's partial (R | r).
template <typename T, int D, int M, bool HAS_O>
__global__ void __launch_bounds__(kThreads)
ncb_query_kernel(const T* __restrict__ Q, const T* __restrict__ O, const T* __restrict__ G,
                 const float* __restrict__ totals, T* __restrict__ dQ, float* __restrict__ ragg,
                 int N, int spans, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP;
    extern __shared__ float smem[];
    float* Ss = smem;             // [D][MP]
    float* Zs = Ss + D * MP;      // [D]
    float* qs = Zs + D;           // [L][DP] phi(Q)
    float* gs = qs + L * DP;      // [L][MP] G, then gn
    float* os = gs + L * MP;      // [L][MP] O
    float* dens = os + L * MP;    // [L]
    float* gds = dens + L;        // [L]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const T* Qh = Q + (size_t)bh * N * D;
    const T* Gh = G + (size_t)bh * N * M;
    T* dQh = dQ + (size_t)bh * N * D;
    load_state<D, M>(Ss, Zs, totals + (size_t)bh * C::W, nullptr, nullptr);
    Frag<D, M> racc;  // sum_i phi(Q_i) gn_i^T over the span
    racc.zero();
    float rsum = 0.f;  // thread d < D: sum_i phi(Q_i)_d gd_i
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(qs, Qh + (size_t)c0 * D, rows, Phi());
        load_tile<L, M, MP>(gs, Gh + (size_t)c0 * M, rows, Ident());
        if (HAS_O) load_tile<L, M, MP>(os, O + ((size_t)bh * N + c0) * M, rows, Ident());
        __syncthreads();
        for (int i = warp; i < L; i += kThreads / 32) {  // den_i = phi(Q_i) . Z
            float a = 0.f;
            for (int d = lane; d < D; d += 32) a = fmaf(qs[i * DP + d], Zs[d], a);
#pragma unroll
            for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) dens[i] = i < rows ? a : 1.f;
        }
        if (!HAS_O) {  // O = phi(Q) S / den
            __syncthreads();
            Frag<L, M> o;
            o.zero();
            o.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int e) { return Ss[d * MP + e]; });
            o.each([&](int i, int e, float x) { os[i * MP + e] = x / dens[i]; });
        }
        __syncthreads();
        for (int i = warp; i < L; i += kThreads / 32) {  // gd_i, gn_i
            const float inv = 1.f / dens[i];
            float a = 0.f;
            for (int e = lane; e < M; e += 32) {
                const float gv = gs[i * MP + e];
                a = fmaf(gv, os[i * MP + e], a);
                gs[i * MP + e] = gv * inv;
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) gds[i] = i < rows ? -a * inv : 0.f;
        }
        __syncthreads();
        {   // dphi(Q_i) = S gn_i + Z gd_i, then phi'(Q) = min(phi(Q), 1)
            Frag<L, D> dq;
            dq.zero();
            dq.template mac<M>([&](int i, int e) { return gs[i * MP + e]; },
                               [&](int e, int d) { return Ss[d * MP + e]; });
            dq.each([&](int i, int d, float x) {
                if (i < rows) {
                    const float f = qs[i * DP + d];
                    dQh[(size_t)(c0 + i) * D + d] = from_f<T>((x + Zs[d] * gds[i]) * dphi_from_phi(f));
                }
            });
        }
        // R += phi(Q)^T gn, r += phi(Q)^T gd over this chunk (rows >= `rows` hold zeros)
        racc.template mac<L>([&](int d, int i) { return qs[i * DP + d]; },
                             [&](int i, int e) { return gs[i * MP + e]; });
        if (threadIdx.x < D)
            for (int i = 0; i < rows; ++i) rsum = fmaf(qs[i * DP + threadIdx.x], gds[i], rsum);
    }
    float* out = ragg + ((size_t)bh * spans + s) * C::W;
    racc.each([&](int d, int e, float x) { out[d * M + e] = x; });
    if (threadIdx.x < D) out[D * M + threadIdx.x] = rsum;
}

// Key side over one span: dK = (R V + r) * phi'(K), dV = phi(K) R.
template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
ncb_key_kernel(const T* __restrict__ K, const T* __restrict__ V, const float* __restrict__ rtot,
               T* __restrict__ dK, T* __restrict__ dV, int N, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP;
    extern __shared__ float smem[];
    float* Rs = smem;           // [D][MP]
    float* rs = Rs + D * MP;    // [D]
    float* ks = rs + D;         // [L][DP] phi(K)
    float* vs = ks + L * DP;    // [L][MP]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const T* Kh = K + (size_t)bh * N * D;
    const T* Vh = V + (size_t)bh * N * M;
    T* dKh = dK + (size_t)bh * N * D;
    T* dVh = dV + (size_t)bh * N * M;
    load_state<D, M>(Rs, rs, rtot + (size_t)bh * C::W, nullptr, nullptr);
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(ks, Kh + (size_t)c0 * D, rows, Phi());
        load_tile<L, M, MP>(vs, Vh + (size_t)c0 * M, rows, Ident());
        __syncthreads();
        {
            Frag<L, D> dk;
            dk.zero();
            dk.template mac<M>([&](int j, int e) { return vs[j * MP + e]; },
                               [&](int e, int d) { return Rs[d * MP + e]; });
            dk.each([&](int j, int d, float x) {
                if (j < rows)
                    dKh[(size_t)(c0 + j) * D + d] = from_f<T>((x + rs[d]) * dphi_from_phi(ks[j * DP + d]));
            });
        }
        {
            Frag<L, M> dv;
            dv.zero();
            dv.template mac<D>([&](int j, int d) { return ks[j * DP + d]; },
                               [&](int d, int e) { return Rs[d * MP + e]; });
            dv.each([&](int j, int e, float x) {
                if (j < rows) dVh[(size_t)(c0 + j) * M + e] = from_f<T>(x);
            });
        }
    }
}

template <int D, int M>
struct NcbSmem {
    using C = Cfg<D, M>;
    static constexpr size_t query =
        sizeof(float) * (D * C::MP + D + C::L * C::DP + 2 * C::L * C::MP + 2 * C::L);
    static constexpr size_t key = sizeof(float) * (D * C::MP + D + C::L * C::DP + C::L * C::MP);
};

}  // namespace ffma

template <typename T, int D, int M>
cudaError_t noncausal_backward(const LaunchCtx& c, const T* Q, const T* K, const T* V, const T* O,
                               const T* G, T* dQ, T* dK, T* dV, int BH, int N) {
    using namespace ffma;
    using C = Cfg<D, M>;
    int spans, span_len;
    choose_spans(BH, N, C::L, c.num_sms, &spans, &span_len);
    const size_t part = (size_t)BH * spans * C::W, tot = (size_t)BH * C::W;
    float* ws = nullptr;
    LA_TRY(scratch_alloc(c, (void**)&ws, plan::ffma_noncausal_backward(BH, N, D, M, c.num_sms)));
    float* sagg = ws;
    float* stot = sagg + part;
    float* ragg = stot + tot;
    float* rtot = ragg + part;
    const unsigned scan_grid = (unsigned)((tot + 255) / 256);
    cudaError_t e = cudaSuccess;
    do {
        if ((e = allow_smem(span_aggregate_kernel<T, D, M>, Smem<D, M>::agg))) break;
        span_aggregate_kernel<T, D, M><<<dim3(BH, spans), kThreads, Smem<D, M>::agg, c.stream>>>(
            K, V, sagg, N, spans, span_len);
        span_scan_kernel<<<scan_grid, 256, 0, c.stream>>>(sagg, nullptr, nullptr, stot, BH, spans, D,
                                                          M, 0);
        if (O) {
            auto kq = ncb_query_kernel<T, D, M, true>;
            if ((e = allow_smem(kq, NcbSmem<D, M>::query))) break;
            kq<<<dim3(BH, spans), kThreads, NcbSmem<D, M>::query, c.stream>>>(Q, O, G, stot, dQ, ragg,
                                                                               N, spans, span_len);
        } else {
            auto kq = ncb_query_kernel<T, D, M, false>;
            if ((e = allow_smem(kq, NcbSmem<D, M>::query))) break;
            kq<<<dim3(BH, spans), kThreads, NcbSmem<D, M>::query, c.stream>>>(Q, O, G, stot, dQ, ragg,
                                                                               N, spans, span_len);
        }
        span_scan_kernel<<<scan_grid, 256, 0, c.stream>>>(ragg, nullptr, nullptr, rtot, BH, spans, D,
                                                          M, 0);
        if ((e = allow_smem(ncb_key_kernel<T, D, M>, NcbSmem<D, M>::key))) break;
        ncb_key_kernel<T, D, M><<<dim3(BH, spans), kThreads, NcbSmem<D, M>::key, c.stream>>>(
            K, V, rtot, dK, dV, N, span_len);
        note_launch(5);
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, ws);
    return e;
}

}  // namespace la
