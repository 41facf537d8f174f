// noncausal_ffma.cuh -- non-causal linear attention phi(Q)(phi(K)^T V) / phi(Q) sum phi(K)
// ("Transformers are RNNs", section 二, eq. linear): per-span aggregates of
// (phi(K)^T V | sum phi(K)), reduced in span order to the head totals S, Z,
// then every query row reads the same S, Z.
#pragma once

#include "causal_ffma.cuh"

namespace la {
namespace ffma {

template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
noncausal_out_kernel(const T* __restrict__ Q, T* __restrict__ O, const float* __restrict__ totals,
                     int N, int span_len) {
    using C = Cfg<D, M>;
    constexpr int L = C::L, DP = C::DP, MP = C::MP;
    extern __shared__ float smem[];
    float* Ss = smem;           // [D][MP]
    float* Zs = Ss + D * MP;    // [D]
    float* qs = Zs + D;         // [L][DP]
    float* dens = qs + L * DP;  // [L]
    const int bh = blockIdx.x, s = blockIdx.y;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    const T* Qh = Q + (size_t)bh * N * D;
    T* Oh = O + (size_t)bh * N * M;
    load_state<D, M>(Ss, Zs, totals + (size_t)bh * C::W, nullptr, nullptr);
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_tile<L, D, DP>(qs, Qh + (size_t)c0 * D, rows, Phi());
        __syncthreads();
        {
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            for (int i = warp; i < L; i += kThreads / 32) {
                float a = 0.f;
                for (int d = lane; d < D; d += 32) a = fmaf(qs[i * DP + d], Zs[d], a);
#pragma unroll
                for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                if (lane == 0) dens[i] = a;
            }
        }
        __syncthreads();
        Frag<L, M> o;
        o.zero();
        o.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                          [&](int d, int e) { return Ss[d * MP + e]; });
        o.each([&](int i, int e, float x) {
            if (i < rows) Oh[(size_t)(c0 + i) * M + e] = from_f<T>(x / dens[i]);
        });
    }
}

}  // namespace ffma

template <typename T, int D, int M>
cudaError_t noncausal_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O,
                              int BH, int N) {
    using namespace ffma;
    using C = Cfg<D, M>;
    int spans, span_len;
    choose_spans(BH, N, C::L, c.num_sms, &spans, &span_len);
    float* ws = nullptr;
    const size_t agg_words = (size_t)BH * spans * C::W;
    LA_TRY(scratch_alloc(c, (void**)&ws, plan::ffma_noncausal_forward(BH, N, D, M, c.num_sms)));
    float* agg = ws;
    float* totals = ws + agg_words;
    cudaError_t e = cudaSuccess;
    do {
        if ((e = allow_smem(span_aggregate_kernel<T, D, M>, Smem<D, M>::agg))) break;
        span_aggregate_kernel<T, D, M><<<dim3(BH, spans), kThreads, Smem<D, M>::agg, c.stream>>>(
            K, V, agg, N, spans, span_len);
        const size_t n = (size_t)BH * C::W;
        span_scan_kernel<<<(unsigned)((n + 255) / 256), 256, 0, c.stream>>>(
            agg, nullptr, nullptr, totals, BH, spans, D, M, 0);
        const size_t smem = sizeof(float) * (D * C::MP + D + C::L * C::DP + C::L);
        if ((e = allow_smem(noncausal_out_kernel<T, D, M>, smem))) break;
        noncausal_out_kernel<T, D, M><<<dim3(BH, spans), kThreads, smem, c.stream>>>(
            Q, O, totals, N, span_len);
        note_launch(3);
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, ws);
    return e;
}

}  // namespace la
