// poly_ffma.cu -- attention with the degree-2 polynomial similarity
// sim(q, k) = (q^T k)^2 in its linear form, on the CUDA cores.
//
// "【论文解读】Transformers are RNNs" section 二 (3) expands (x^T y)^2 into the
// inner product of the explicit feature maps phi(x) = (x_a x_b), C = D^2
// features, so that
//     V'_i = phi(Q_i)^T S / phi(Q_i)^T Z,  S = sum_j phi(K_j) V_j^T,  Z = sum_j phi(K_j)
// with the sums over j <= i (causal, section 三) or over all j, at a cost of
// O(N D^2 M).  x_a x_b is symmetric in (a, b), so this implementation keeps
// the P = D (D + 1) / 2 features with a <= b and weights the key side by 2
// where a < b: sum_{a<=b} (q_a q_b)(w_ab k_a k_b) = (q . k)^2 exactly.
//
// Work split: the P feature rows of the state are cut into NSL slices; a CTA
// owns one (head, span, slice).  A first pass forms each span's aggregate of
// its slice ((sum phi(K) V^T | sum phi(K)) over the span), a scan over spans
// gives each span its starting state (causal) or the totals (non-causal), and
// the main pass walks the span's chunks: it adds phi(Q) [S | Z] of its slice
// to an fp32 accumulator of numerators and denominators (one atomic add per
// element and slice), then, when causal, updates its slice of the state.  The
// slice-0 CTA also adds the intra-chunk terms sum_{j<=i, same chunk}
// (q_i . k_j)^2 [V_j | 1].  A last kernel divides and stores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "la_common.cuh"
#include "la_launch.h"
#include "la_plan.h"

namespace la {
namespace poly {

constexpr int kThreads = 256;
constexpr int D = 32;                       // head size of the queries and keys
constexpr int P = D * (D + 1) / 2;          // distinct features (a <= b)
constexpr int NSL = plan::kPolySlices;      // feature slices
constexpr int PS = P / NSL;                 // features per slice
constexpr int L = 64;                       // chunk length
static_assert(P % NSL == 0 && PS % 16 == 0, "slices of whole 16-row blocks");

template <int M>
struct Lay {
    static constexpr int MP = M + 1, PP = PS + 1, DP = D + 1, LP = L + 1;
    // shared memory, in floats
    static constexpr int S = 0;                   // [PS][MP] state slice, column M = Z
    static constexpr int FQ = S + PS * MP;        // [L][PP] phi(Q) slice
    static constexpr int FK = FQ + L * PP;        // [L][PP] weighted phi(K) slice
    static constexpr int QS = FK + L * PP;        // [L][DP]
    static constexpr int KS = QS + L * DP;        // [L][DP]
    static constexpr int VS = KS + L * DP;        // [L][MP] V, column M = 1
    static constexpr int PM = VS + L * MP;        // [L][LP] intra-chunk weights (slice 0)
    static constexpr int AB = PM + L * LP;        // [PS] packed (a, b) of the slice's features
    static constexpr int FLOATS = AB + PS;
    static constexpr size_t BYTES = sizeof(float) * FLOATS;
};

// Register tile of 256 threads (16 x 16): acc[r][c] for rows ty + 16 r, cols tx + 16 c.
template <int R, int C>
struct Tile {
    float v[R / 16][C / 16];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int a = 0; a < R / 16; ++a)
#pragma unroll
            for (int b = 0; b < C / 16; ++b) v[a][b] = 0.f;
    }
    template <int KD, class FA, class FB>
    __device__ __forceinline__ void mac(FA A, FB B) {
        const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll 4
        for (int k = 0; k < KD; ++k) {
            float av[R / 16], bv[C / 16];
#pragma unroll
            for (int a = 0; a < R / 16; ++a) av[a] = A(ty + 16 * a, k);
#pragma unroll
            for (int b = 0; b < C / 16; ++b) bv[b] = B(k, tx + 16 * b);
#pragma unroll
            for (int a = 0; a < R / 16; ++a)
#pragma unroll
                for (int b = 0; b < C / 16; ++b) v[a][b] = fmaf(av[a], bv[b], v[a][b]);
        }
    }
    template <class F>
    __device__ __forceinline__ void each(F f) {
        const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
        for (int a = 0; a < R / 16; ++a)
#pragma unroll
            for (int b = 0; b < C / 16; ++b) f(ty + 16 * a, tx + 16 * b, v[a][b]);
    }
};

// (a, b) of feature p (a <= b, a-major), packed a | b << 8.
__device__ __forceinline__ void fill_pairs(float* ab, int slice) {
    for (int t = threadIdx.x; t < PS; t += kThreads) {
        int p = slice * PS + t, a = 0;
        while (p >= D - a) {
            p -= D - a;
            ++a;
        }
        ab[t] = __int_as_float(a | ((a + p) << 8));
    }
}

// Loads `rows` rows of a [*, C] tile (row stride CP), zero beyond; for V the
// extra column C is 1 on valid rows.
template <typename T, int C, int CP, bool ONE_COL>
__device__ __forceinline__ void load_rows(float* dst, const T* __restrict__ src, int rows) {
    for (int t = threadIdx.x; t < L * C; t += kThreads) {
        const int r = t / C, c = t - r * C;
        dst[r * CP + c] = r < rows ? to_f(src[(size_t)r * C + c]) : 0.f;
    }
    if (ONE_COL)
        for (int r = threadIdx.x; r < L; r += kThreads) dst[r * CP + C] = r < rows ? 1.f : 0.f;
}

// phi slice of the rows in xs: f[i][t] = x_a x_b (times 2 for a < b when WEIGHT).
template <bool WEIGHT>
__device__ __forceinline__ void feature_slice(float* f, const float* xs, const float* ab) {
    for (int t = threadIdx.x; t < L * PS; t += kThreads) {
        const int i = t / PS, c = t - i * PS;
        const int pk = __float_as_int(ab[c]), a = pk & 0xFF, b = pk >> 8;
        const float w = WEIGHT && a != b ? 2.f : 1.f;
        f[i * (PS + 1) + c] = w * xs[i * (D + 1) + a] * xs[i * (D + 1) + b];
    }
}

// Aggregate of a span's slice: (sum_j phi(K_j) [V_j | 1]^T), [PS][M + 1].
template <typename T, int M>
__global__ void __launch_bounds__(kThreads)
poly_aggregate_kernel(const T* __restrict__ K, const T* __restrict__ V, float* __restrict__ agg,
                      int N, int spans, int span_len) {
    using Ly = Lay<M>;
    extern __shared__ float sm[];
    const int bh = blockIdx.x, s = blockIdx.y, sl = blockIdx.z;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    float* fk = sm + Ly::FK;
    float* ks = sm + Ly::KS;
    float* vs = sm + Ly::VS;
    float* ab = sm + Ly::AB;
    fill_pairs(ab, sl);
    Tile<PS, M> acc;
    acc.zero();
    float z = 0.f;  // thread t < PS: sum of its feature over the span
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_rows<T, D, Ly::DP, false>(ks, K + ((size_t)bh * N + c0) * D, rows);
        load_rows<T, M, Ly::MP, true>(vs, V + ((size_t)bh * N + c0) * M, rows);
        __syncthreads();
        feature_slice<true>(fk, ks, ab);
        __syncthreads();
        acc.template mac<L>([&](int p, int j) { return fk[j * Ly::PP + p]; },
                            [&](int j, int e) { return vs[j * Ly::MP + e]; });
        for (int t = threadIdx.x; t < PS; t += kThreads)
            for (int j = 0; j < L; ++j) z += fk[j * Ly::PP + t];
    }
    float* out = agg + (((size_t)bh * spans + s) * NSL + sl) * PS * Ly::MP;
    acc.each([&](int p, int e, float x) { out[p * Ly::MP + e] = x; });
    for (int t = threadIdx.x; t < PS; t += kThreads) out[t * Ly::MP + M] = z;
}

// In place over spans: exclusive prefix (causal) or every span's slot set to
// the total (non-causal).
static __global__ void poly_scan_kernel(float* __restrict__ agg, int BH, int spans, int words,
                                        int causal) {
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)BH * words) return;
    const int bh = (int)(idx / words), w = (int)(idx - (size_t)bh * words);
    float run = 0.f;
    for (int s = 0; s < spans; ++s) {
        float* p = agg + ((size_t)bh * spans + s) * words + w;
        const float x = *p;
        if (causal) *p = run;
        run += x;
    }
    if (!causal)
        for (int s = 0; s < spans; ++s) agg[((size_t)bh * spans + s) * words + w] = run;
}

// One (head, span, slice): numerators and denominators into acc [BH][N][M + 1].
template <typename T, int M, bool CAUSAL>
__global__ void __launch_bounds__(kThreads)
poly_main_kernel(const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                 const float* __restrict__ prefix, float* __restrict__ acc, int N, int spans,
                 int span_len) {
    using Ly = Lay<M>;
    constexpr int MP = Ly::MP, PP = Ly::PP, DP = Ly::DP, LP = Ly::LP;
    extern __shared__ float sm[];
    const int bh = blockIdx.x, s = blockIdx.y, sl = blockIdx.z;
    const int n0 = s * span_len, n1 = min(N, n0 + span_len);
    float* Ss = sm + Ly::S;
    float* fq = sm + Ly::FQ;
    float* fk = sm + Ly::FK;
    float* qs = sm + Ly::QS;
    float* ks = sm + Ly::KS;
    float* vs = sm + Ly::VS;
    float* pm = sm + Ly::PM;
    float* ab = sm + Ly::AB;
    fill_pairs(ab, sl);
    {
        const float* src = prefix + (((size_t)bh * spans + s) * NSL + sl) * PS * MP;
        for (int t = threadIdx.x; t < PS * MP; t += kThreads) Ss[t] = src[t];
    }
    float* acc_h = acc + (size_t)bh * N * MP;
    for (int c0 = n0; c0 < n1; c0 += L) {
        const int rows = min(L, n1 - c0);
        __syncthreads();
        load_rows<T, D, DP, false>(qs, Q + ((size_t)bh * N + c0) * D, rows);
        if (CAUSAL) {
            load_rows<T, D, DP, false>(ks, K + ((size_t)bh * N + c0) * D, rows);
            load_rows<T, M, MP, true>(vs, V + ((size_t)bh * N + c0) * M, rows);
        }
        __syncthreads();
        feature_slice<false>(fq, qs, ab);
        if (CAUSAL) feature_slice<true>(fk, ks, ab);
        if (CAUSAL && sl == 0) {  // intra-chunk weights (q_i . k_j)^2, j <= i
            Tile<L, L> w;
            w.zero();
            w.template mac<D>([&](int i, int d) { return qs[i * DP + d]; },
                              [&](int d, int j) { return ks[j * DP + d]; });
            w.each([&](int i, int j, float x) { pm[i * LP + j] = j <= i ? x * x : 0.f; });
        }
        __syncthreads();
        {   // phi(Q) [S | Z] over this slice (+ the intra-chunk terms on slice 0)
            Tile<L, M> o;
            o.zero();
            o.template mac<PS>([&](int i, int p) { return fq[i * PP + p]; },
                               [&](int p, int e) { return Ss[p * MP + e]; });
            if (CAUSAL && sl == 0)
                o.template mac<L>([&](int i, int j) { return pm[i * LP + j]; },
                                  [&](int j, int e) { return vs[j * MP + e]; });
            o.each([&](int i, int e, float x) {
                if (i < rows) atomicAdd(acc_h + (size_t)(c0 + i) * MP + e, x);
            });
            const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
            for (int i = warp; i < rows; i += kThreads / 32) {  // the denominators
                float a = 0.f;
                for (int p = lane; p < PS; p += 32) a = fmaf(fq[i * PP + p], Ss[p * MP + M], a);
                if (CAUSAL && sl == 0)
                    for (int j = lane; j < L; j += 32) a += pm[i * LP + j];
#pragma unroll
                for (int o2 = 16; o2; o2 >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o2);
                if (lane == 0) atomicAdd(acc_h + (size_t)(c0 + i) * MP + M, a);
            }
        }
        if (CAUSAL) {  // S += phi(K)^T [V | 1] over this slice
            __syncthreads();
            Tile<PS, M> u;
            u.zero();
            u.template mac<L>([&](int p, int j) { return fk[j * PP + p]; },
                              [&](int j, int e) { return vs[j * MP + e]; });
            u.each([&](int p, int e, float x) { Ss[p * MP + e] += x; });
            for (int t = threadIdx.x; t < PS; t += kThreads) {
                float z = 0.f;
                for (int j = 0; j < L; ++j) z += fk[j * PP + t];
                Ss[t * MP + M] += z;
            }
        }
    }
}

template <typename T, int M>
__global__ void poly_divide_kernel(const float* __restrict__ acc, T* __restrict__ O, size_t rows) {
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * M) return;
    const size_t r = idx / M;
    const int e = (int)(idx - r * M);
    O[idx] = from_f<T>(acc[r * (M + 1) + e] / acc[r * (M + 1) + M]);
}

}  // namespace poly

template <typename T, int M>
cudaError_t poly2_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O, int BH,
                          int N, bool causal) {
    using namespace poly;
    using Ly = Lay<M>;
    int spans = 1, span_len = N;
    plan::poly_spans(BH, N, c.num_sms, &spans, &span_len);
    const size_t words = (size_t)NSL * PS * Ly::MP;  // one span's state, all slices
    const size_t agg_bytes = sizeof(float) * (size_t)BH * spans * words;
    const size_t acc_bytes = sizeof(float) * (size_t)BH * N * Ly::MP;
    char* ws = nullptr;
    cudaError_t e = scratch_alloc(c, reinterpret_cast<void**>(&ws), plan::poly2_scratch(BH, N, M, c.num_sms));
    if (e != cudaSuccess) return e;
    float* agg = reinterpret_cast<float*>(ws);
    float* acc = reinterpret_cast<float*>(ws + plan::up256(agg_bytes));
    do {
        auto ka = poly_aggregate_kernel<T, M>;
        auto km = causal ? poly_main_kernel<T, M, true> : poly_main_kernel<T, M, false>;
        if ((e = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly::BYTES)) ||
            (e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly::BYTES)))
            break;
        if ((e = cudaMemsetAsync(acc, 0, acc_bytes, c.stream))) break;
        const dim3 grid(BH, spans, NSL);
        ka<<<grid, kThreads, Ly::BYTES, c.stream>>>(K, V, agg, N, spans, span_len);
        const size_t n = (size_t)BH * words;
        poly_scan_kernel<<<(unsigned)((n + 255) / 256), 256, 0, c.stream>>>(agg, BH, spans, (int)words,
                                                                           causal ? 1 : 0);
        km<<<grid, kThreads, Ly::BYTES, c.stream>>>(Q, K, V, agg, acc, N, spans, span_len);
        const size_t outs = (size_t)BH * N * M;
        poly_divide_kernel<T, M><<<(unsigned)((outs + 255) / 256), 256, 0, c.stream>>>(acc, O,
                                                                                     (size_t)BH * N);
        note_launch(4);
        e = cudaGetLastError();
    } while (0);
    scratch_free(c, ws);
    return e;
}

#define LA_INST_POLY(T, M)                                                                     \
    template cudaError_t poly2_forward<T, M>(const LaunchCtx&, const T*, const T*, const T*, T*, \
                                             int, int, bool);
LA_INST_POLY(float, 32) LA_INST_POLY(float, 64)
LA_INST_POLY(__nv_bfloat16, 32) LA_INST_POLY(__nv_bfloat16, 64)

}  // namespace la
