// la_common.cuh -- device helpers shared by the linear-attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

// phi(x) = elu(x) + 1 with alpha = 1: x + 1 for x > 0, e^x otherwise
// ("Transformers are RNNs", section 特征映射, eq. elu).
__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }

// phi'(x) = 1 for x > 0 and e^x = phi(x) otherwise, so phi'(x) = min(phi(x), 1)
// (phi(x) > 1 exactly when x > 0).
__device__ __forceinline__ float dphi_from_phi(float f) { return fminf(f, 1.f); }

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Block-level register-tiled product for 256 threads arranged 16 x 16:
// acc[a][b] += sum_k A(ty + 16a, k) * B(k, tx + 16b) for an R x C output.
// Strided ownership keeps shared-memory reads of B conflict-free.
template <int R, int C>
struct Frag {
    static constexpr int TR = R / 16;
    static constexpr int TC = C / 16;
    float v[TR][TC];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int a = 0; a < TR; ++a)
#pragma unroll
            for (int b = 0; b < TC; ++b) v[a][b] = 0.f;
    }
    template <int KD, class FA, class FB>
    __device__ __forceinline__ void mac(FA A, FB B) {
        const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
        for (int k = 0; k < KD; ++k) {
            float av[TR], bv[TC];
#pragma unroll
            for (int a = 0; a < TR; ++a) av[a] = A(ty + 16 * a, k);
#pragma unroll
            for (int b = 0; b < TC; ++b) bv[b] = B(k, tx + 16 * b);
#pragma unroll
            for (int a = 0; a < TR; ++a)
#pragma unroll
                for (int b = 0; b < TC; ++b) v[a][b] = fmaf(av[a], bv[b], v[a][b]);
        }
    }
    template <class F>
    __device__ __forceinline__ void each(F f) {
        const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
        for (int a = 0; a < TR; ++a)
#pragma unroll
            for (int b = 0; b < TC; ++b) f(ty + 16 * a, tx + 16 * b, v[a][b]);
    }
};

}  // namespace la
