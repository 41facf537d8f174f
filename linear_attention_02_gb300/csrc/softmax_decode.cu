// softmax_decode.cu -- one decode step of standard softmax attention with a KV
// cache, the comparator of the recurrent linear-attention step.
//
// Standard Transformer inference ("Transformer与RNN的深层联结", section 2)
// appends the step's k, v to the cache and attends over every cached position:
//     out = softmax(q K^T / sqrt(D)) V
// (the scaled dot product of "Transformers are RNNs", section 一, eq. softmax).
// Its cost grows with the cache, where the linear-attention step reads a
// fixed D x M state: this kernel is here to measure that difference on the
// same hardware.  It is bandwidth-bound: every cached key and value row is
// read once per step.
//
// Layout: a head's cache rows are contiguous, K_cache [BH][T_max][D],
// V_cache [BH][T_max][M] (M = D).  Each CTA takes a range of positions of one
// head; a lane group of LR lanes holds one row (16 bytes a lane) and a warp
// works on 32 / LR rows at a time, eight rows per lane group in flight.  Scores
// are kept in base 2 (q pre-scaled by log2(e) / sqrt(D)), and each lane group
// keeps a running maximum, a running sum of weights and its slice of the
// weighted value sum (the online form of the max-subtracted softmax).  The
// groups merge by shuffles, the warps through shared memory, and the ranges
// of a head in a second small kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "la_common.cuh"
#include "la_launch.h"
#include "la_plan.h"

namespace la {
namespace {

constexpr int kSdThreads = 256;
constexpr int kSdUnroll = 8;

template <typename T, int D>
struct SdShape {
    static constexpr int EPL = 16 / static_cast<int>(sizeof(T));  // elements per lane (16 bytes)
    static constexpr int LR = D / EPL;                              // lanes per row
    static constexpr int RPW = 32 / LR;                             // rows per warp step
    static constexpr int WARPS = kSdThreads / 32;
    static_assert(LR >= 1 && LR <= 32 && 32 % LR == 0, "row split");
};

template <typename T, int EPL>
__device__ __forceinline__ void unpack(const uint4& u, float (&x)[EPL]);
template <>
__device__ __forceinline__ void unpack<__nv_bfloat16, 8>(const uint4& u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void unpack<float, 4>(const uint4& u, float (&x)[4]) {
    x[0] = __uint_as_float(u.x);
    x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z);
    x[3] = __uint_as_float(u.w);
}

// Merges the running softmax state (m2, l2, a2) into (m, l, a): maxima in base 2.
template <int EPL>
__device__ __forceinline__ void merge(float& m, float& l, float (&a)[EPL], float m2, float l2,
                                      const float (&a2)[EPL]) {
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;  // both empty
    const float f1 = exp2f(m - mn), f2 = exp2f(m2 - mn);
    l = l * f1 + l2 * f2;
#pragma unroll
    for (int i = 0; i < EPL; ++i) a[i] = a[i] * f1 + a2[i] * f2;
    m = mn;
}

// Range `blockIdx.y` of head `blockIdx.x`: positions [j0, j1) of the T_len + 1
// (position T_len is the step's own k, v, written into the cache here).
template <typename T, int D>
__global__ void __launch_bounds__(kSdThreads)
softmax_decode_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      T* __restrict__ Kc, T* __restrict__ Vc, int T_len, int T_max, int split_len,
                      float* __restrict__ part) {
    using Sh = SdShape<T, D>;
    constexpr int EPL = Sh::EPL, LR = Sh::LR, RPW = Sh::RPW, WARPS = Sh::WARPS;
    constexpr int STEP = WARPS * RPW;  // rows per CTA step
    __shared__ float sm_m[WARPS], sm_l[WARPS];
    __shared__ float sm_a[WARPS][D];
    const int bh = blockIdx.x, sp = blockIdx.y, splits = gridDim.y;
    const int total = T_len + 1;
    const int j0 = sp * split_len, j1 = min(total, j0 + split_len);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / LR, c = lane % LR;  // row within the warp step, 16-byte chunk of the row
    const size_t base = static_cast<size_t>(bh) * T_max * D + static_cast<size_t>(c) * EPL;
    const uint4* K4 = reinterpret_cast<const uint4*>(Kc + base);
    const uint4* V4 = reinterpret_cast<const uint4*>(Vc + base);
    constexpr int ROW4 = D / EPL;  // uint4 per row

    float qv[EPL];
    {
        const uint4 u = *reinterpret_cast<const uint4*>(q + static_cast<size_t>(bh) * D + c * EPL);
        unpack<T, EPL>(u, qv);
        const float sc = 1.4426950408889634f / sqrtf(static_cast<float>(D));  // log2(e) / sqrt(D)
#pragma unroll
        for (int i = 0; i < EPL; ++i) qv[i] *= sc;
    }
    const uint4 knew = *reinterpret_cast<const uint4*>(k + static_cast<size_t>(bh) * D + c * EPL);
    const uint4 vnew = *reinterpret_cast<const uint4*>(v + static_cast<size_t>(bh) * D + c * EPL);

    float m = -INFINITY, l = 0.f, acc[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] = 0.f;

    // The loop bound is the warp's (wb), the same for all of its lanes, so every
    // lane takes part in every shuffle below; rows at or past j1 are skipped
    // after the shuffle.
    for (int wb = j0 + warp * RPW; wb < j1; wb += kSdUnroll * STEP) {
        const int jb = wb + slot;
        uint4 kr[kSdUnroll], vr[kSdUnroll];
#pragma unroll
        for (int u = 0; u < kSdUnroll; ++u) {  // every load of this step first
            const int j = jb + u * STEP;
            if (j < T_len && j < j1) {
                kr[u] = __ldcs(K4 + static_cast<size_t>(j) * ROW4);
                vr[u] = __ldcs(V4 + static_cast<size_t>(j) * ROW4);
            } else {
                kr[u] = knew;
                vr[u] = vnew;
            }
        }
#pragma unroll
        for (int u = 0; u < kSdUnroll; ++u) {
            const int j = jb + u * STEP;
            float kx[EPL], vx[EPL];
            unpack<T, EPL>(kr[u], kx);
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) s = fmaf(qv[i], kx[i], s);
#pragma unroll
            for (int o = LR / 2; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (j >= j1) continue;  // uniform over the lane group
            if (j == T_len) {       // the step's own row goes into the cache
                const_cast<uint4*>(K4)[static_cast<size_t>(j) * ROW4] = knew;
                const_cast<uint4*>(V4)[static_cast<size_t>(j) * ROW4] = vnew;
            }
            unpack<T, EPL>(vr[u], vx);
            const float mn = fmaxf(m, s);
            const float f = exp2f(m - mn), p = exp2f(s - mn);
            l = l * f + p;
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc[i] = fmaf(p, vx[i], acc[i] * f);
            m = mn;
        }
    }
    // lane groups of the warp (lanes with the same chunk c)
#pragma unroll
    for (int o = LR; o < 32; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        float a2[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) a2[i] = __shfl_xor_sync(0xffffffffu, acc[i], o);
        merge<EPL>(m, l, acc, m2, l2, a2);
    }
    if (lane < LR) {
#pragma unroll
        for (int i = 0; i < EPL; ++i) sm_a[warp][c * EPL + i] = acc[i];
        if (lane == 0) {
            sm_m[warp] = m;
            sm_l[warp] = l;
        }
    }
    __syncthreads();
    float* out = part + (static_cast<size_t>(bh) * splits + sp) * (D + 2);
    for (int e = threadIdx.x; e < D; e += kSdThreads) {
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) mm = fmaxf(mm, sm_m[w]);
        float ll = 0.f, aa = 0.f;
        if (mm != -INFINITY) {
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float f = exp2f(sm_m[w] - mm);
                ll += sm_l[w] * f;
                aa += sm_a[w][e] * f;
            }
        }
        out[2 + e] = aa;
        if (e == 0) {
            out[0] = mm;
            out[1] = ll;
        }
    }
}

// out[bh] = the ranges of head bh merged: sum a 2^(m - M) / sum l 2^(m - M).
template <int D>
__global__ void softmax_decode_combine(const float* __restrict__ part, float* __restrict__ out,
                                       int splits) {
    const int bh = blockIdx.x, e = threadIdx.x;
    const float* p = part + static_cast<size_t>(bh) * splits * (D + 2);
    float mm = -INFINITY;
    for (int s = 0; s < splits; ++s) mm = fmaxf(mm, p[s * (D + 2)]);
    float ll = 0.f, aa = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float ms = p[s * (D + 2)];
        if (ms == -INFINITY) continue;
        const float f = exp2f(ms - mm);
        ll += p[s * (D + 2) + 1] * f;
        aa += p[s * (D + 2) + 2 + e] * f;
    }
    out[static_cast<size_t>(bh) * D + e] = aa / ll;
}

}  // namespace

template <typename T, int D>
cudaError_t softmax_decode_step(const LaunchCtx& c, const T* q, const T* k, const T* v, T* Kc,
                                T* Vc, int T_len, int T_max, float* out, int BH) {
    int splits = 1, split_len = 1;
    plan::softmax_decode_split(BH, T_len + 1, c.num_sms, &splits, &split_len);
    float* part = nullptr;
    cudaError_t e = scratch_alloc(c, reinterpret_cast<void**>(&part),
                                  plan::softmax_decode_scratch(BH, T_len + 1, D, c.num_sms));
    if (e != cudaSuccess) return e;
    softmax_decode_kernel<T, D><<<dim3(BH, splits), kSdThreads, 0, c.stream>>>(
        q, k, v, Kc, Vc, T_len, T_max, split_len, part);
    softmax_decode_combine<D><<<BH, D, 0, c.stream>>>(part, out, splits);
    note_launch(2);
    e = cudaGetLastError();
    scratch_free(c, part);
    return e;
}

#define LA_INST_SD(T, D)                                                                         \
    template cudaError_t softmax_decode_step<T, D>(const LaunchCtx&, const T*, const T*, const T*, \
                                                   T*, T*, int, int, float*, int);
LA_INST_SD(float, 32) LA_INST_SD(float, 64) LA_INST_SD(float, 128)
LA_INST_SD(__nv_bfloat16, 32) LA_INST_SD(__nv_bfloat16, 64) LA_INST_SD(__nv_bfloat16, 128)

}  // namespace la
