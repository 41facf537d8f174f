// decode.cu -- one recurrent decode step per head, bandwidth-bound.
//
// RNN form of "Transformers are RNNs" (section 四) in the order of RNN-mode
// inference ("Transformer与RNN的深层联结", section 2): update first,
//   S += phi(k) v^T,  Z += phi(k),
// then read
//   out = phi(q)^T S / phi(q)^T Z.
// The fp32 state S [D][M] is streamed once in and once out with 128-bit
// accesses; the read-out is fused into the same pass over S (each thread
// forms phi(q)_d * S_new[d][e] for its rows and the partial sums are reduced
// with warp shuffles, then across warps in shared memory).  Each thread holds
// 8 rows of four columns where the block allows (128 threads per head at
// D = M = 64; 4 and 16 rows measured slower), and every load of the block
// (S rows, then q, k, Z and v) is issued before any is used, so their latencies
// overlap; Z's update and the denominator are reduced before the first barrier.
#include "la_common.cuh"
#include "la_launch.h"

namespace la {

namespace {

template <int D, int M, int ROWS = 8>
struct DecShape {
    static constexpr int CG = M / 4;  // float4 column groups of a row
    // ROWS rows per thread where the block allows (at least two warps)
    static constexpr int THREADS = CG * D / ROWS > 64 ? CG * D / ROWS : 64;
    static constexpr int RG = THREADS / CG;                             // row groups
    static constexpr int RPT = D / RG;                                  // rows per thread
    static constexpr int WARPS = THREADS / 32;
    static_assert(RPT >= 1 && D % RG == 0 && THREADS % 32 == 0 && CG <= 32, "shape");
};

template <typename T, int D, int M, int ROWS = 8>
__global__ void __launch_bounds__(DecShape<D, M, ROWS>::THREADS)
decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   float* __restrict__ S, float* __restrict__ Z, float* __restrict__ out, int BH) {
    using Sh = DecShape<D, M, ROWS>;
    constexpr int CG = Sh::CG, RG = Sh::RG, RPT = Sh::RPT, WARPS = Sh::WARPS, NT = Sh::THREADS;
    constexpr int ZW = (D + 31) / 32;  // warps holding a row of Z
    static_assert(D <= NT && M <= NT, "one element of q, k, Z and v per thread");
    __shared__ float fq[D], fk[D], vv[M];
    __shared__ float4 red[WARPS][CG];
    __shared__ float red_den[ZW];
    const int bh = blockIdx.x;
    const int t = threadIdx.x;
    const int cg = t % CG, rg = t / CG;
    const int warp = t >> 5, lane = t & 31;
    float4* S4 = reinterpret_cast<float4*>(S + (size_t)bh * D * M);
    // Every load this block needs is issued before any is used: the S rows, then
    // this thread's element of q, k, Z and v, so their latencies overlap.
    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s[r] = S4[(size_t)(rg + r * RG) * CG + cg];
    float qd = 0.f, kd = 0.f, zd = 0.f, vd = 0.f;
    if (t < D) {
        qd = to_f(q[(size_t)bh * D + t]);
        kd = to_f(k[(size_t)bh * D + t]);
        zd = Z[(size_t)bh * D + t];
    }
    if (t < M) vd = to_f(v[(size_t)bh * M + t]);
    // Z += phi(k) and this thread's term of the denominator phi(q) . Z, reduced
    // per warp before the first barrier
    float dpart = 0.f;
    if (t < D) {
        const float a = phi(kd), b = phi(qd);
        fk[t] = a;
        fq[t] = b;
        zd += a;
        Z[(size_t)bh * D + t] = zd;
        dpart = b * zd;
    }
    if (t < M) vv[t] = vd;
    if (warp < ZW) {
#pragma unroll
        for (int o = 16; o; o >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, o);
        if (lane == 0) red_den[warp] = dpart;
    }
    __syncthreads();

    const float4 v4 = make_float4(vv[4 * cg], vv[4 * cg + 1], vv[4 * cg + 2], vv[4 * cg + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int d = rg + r * RG;
        const float a = fk[d], b = fq[d];
        s[r].x = fmaf(a, v4.x, s[r].x);
        s[r].y = fmaf(a, v4.y, s[r].y);
        s[r].z = fmaf(a, v4.z, s[r].z);
        s[r].w = fmaf(a, v4.w, s[r].w);
        S4[(size_t)d * CG + cg] = s[r];
        acc.x = fmaf(b, s[r].x, acc.x);
        acc.y = fmaf(b, s[r].y, acc.y);
        acc.z = fmaf(b, s[r].z, acc.z);
        acc.w = fmaf(b, s[r].w, acc.w);
    }
    // reduce over the row groups held by this warp (lanes cg, cg + CG, ...)
#pragma unroll
    for (int o = CG; o < 32; o <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    }
    if (lane < CG) red[warp][lane] = acc;
    __syncthreads();
    if (t < CG) {
        // warps that hold distinct row groups: each warp covers 32 / CG row groups
        float4 a = red[0][t];
        for (int w = 1; w < WARPS; ++w) {
            const float4 b = red[w][t];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        float den = red_den[0];
#pragma unroll
        for (int w = 1; w < ZW; ++w) den += red_den[w];
        const float inv_den = 1.f / den;
        float4 o4 = make_float4(a.x * inv_den, a.y * inv_den, a.z * inv_den, a.w * inv_den);
        reinterpret_cast<float4*>(out + (size_t)bh * M)[t] = o4;
    }
}

// One retention step per head ("Transformer and Variants" section 1.3.4, in
// the S = sum k v^T convention): S = gamma S + k v^T, then out = S^T q, raw q
// and k, no normaliser.  gamma: gate[bh] (this step's decay of each head) if
// given, else gamma_head[bh % H], else 1.  Same streaming of S as above.
template <typename T, int D, int M, int ROWS = 8>
__global__ void __launch_bounds__(DecShape<D, M, ROWS>::THREADS)
retention_step_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                      const float* __restrict__ gamma_head, const float* __restrict__ gate,
                      float* __restrict__ S, float* __restrict__ out, int H) {
    using Sh = DecShape<D, M, ROWS>;
    constexpr int CG = Sh::CG, RG = Sh::RG, RPT = Sh::RPT, WARPS = Sh::WARPS;
    static_assert(D <= Sh::THREADS && M <= Sh::THREADS, "one element of q, k and v per thread");
    __shared__ float qs[D], ks[D], vv[M];
    __shared__ float4 red[WARPS][CG];
    const int bh = blockIdx.x;
    const int t = threadIdx.x;
    const int cg = t % CG, rg = t / CG;
    const int warp = t >> 5, lane = t & 31;
    float4* S4 = reinterpret_cast<float4*>(S + (size_t)bh * D * M);
    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s[r] = S4[(size_t)(rg + r * RG) * CG + cg];
    const float g = gate ? gate[bh] : (gamma_head ? gamma_head[bh % H] : 1.f);
    if (t < D) {
        qs[t] = to_f(q[(size_t)bh * D + t]);
        ks[t] = to_f(k[(size_t)bh * D + t]);
    }
    if (t < M) vv[t] = to_f(v[(size_t)bh * M + t]);
    __syncthreads();
    const float4 v4 = make_float4(vv[4 * cg], vv[4 * cg + 1], vv[4 * cg + 2], vv[4 * cg + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int d = rg + r * RG;
        const float a = ks[d], b = qs[d];
        s[r].x = fmaf(a, v4.x, g * s[r].x);
        s[r].y = fmaf(a, v4.y, g * s[r].y);
        s[r].z = fmaf(a, v4.z, g * s[r].z);
        s[r].w = fmaf(a, v4.w, g * s[r].w);
        S4[(size_t)d * CG + cg] = s[r];
        acc.x = fmaf(b, s[r].x, acc.x);
        acc.y = fmaf(b, s[r].y, acc.y);
        acc.z = fmaf(b, s[r].z, acc.z);
        acc.w = fmaf(b, s[r].w, acc.w);
    }
#pragma unroll
    for (int o = CG; o < 32; o <<= 1) {
        acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
        acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
        acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
        acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
    }
    if (lane < CG) red[warp][lane] = acc;
    __syncthreads();
    if (t < CG) {
        float4 a = red[0][t];
        for (int w = 1; w < WARPS; ++w) {
            const float4 b = red[w][t];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        reinterpret_cast<float4*>(out + (size_t)bh * M)[t] = a;
    }
}

}  // namespace

template <typename T, int D, int M>
cudaError_t retention_step(const LaunchCtx& c, const T* q, const T* k, const T* v,
                           const float* gamma_head, const float* gate, float* S, float* out, int BH,
                           int H) {
    retention_step_kernel<T, D, M><<<BH, DecShape<D, M>::THREADS, 0, c.stream>>>(q, k, v, gamma_head,
                                                                                 gate, S, out, H);
    note_launch();
    return cudaGetLastError();
}

template <typename T, int D, int M>
cudaError_t decode_step(const LaunchCtx& c, const T* q, const T* k, const T* v, float* S,
                        float* Z, float* out, int BH) {
    decode_step_kernel<T, D, M><<<BH, DecShape<D, M>::THREADS, 0, c.stream>>>(q, k, v, S, Z, out, BH);
    note_launch();
    return cudaGetLastError();
}

#define LA_INST_DEC(T, D, M)                                                                      \
    template cudaError_t decode_step<T, D, M>(const LaunchCtx&, const T*, const T*, const T*,    \
                                              float*, float*, float*, int);                      \
    template cudaError_t retention_step<T, D, M>(const LaunchCtx&, const T*, const T*, const T*, \
                                                 const float*, const float*, float*, float*, int, \
                                                 int);
#define LA_INST_DEC_T(T) \
    LA_INST_DEC(T, 32, 32) LA_INST_DEC(T, 32, 64) LA_INST_DEC(T, 32, 128) \
    LA_INST_DEC(T, 64, 32) LA_INST_DEC(T, 64, 64) LA_INST_DEC(T, 64, 128) \
    LA_INST_DEC(T, 128, 32) LA_INST_DEC(T, 128, 64) LA_INST_DEC(T, 128, 128)
LA_INST_DEC_T(float)
LA_INST_DEC_T(__nv_bfloat16)

}  // namespace la
