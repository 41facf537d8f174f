// noalloc.cu -- la_forward_noncausal_noalloc: the non-causal forward with its
// scratch in a fixed, file-scope device array instead of the library's pool.
//
// Some callers must not allocate device memory while running an op: a host
// framework that plans every byte of device memory ahead of time and hands an
// op only its inputs and outputs, a plugin runtime that forbids allocation
// inside the op, or a latency-critical loop that cannot afford an allocator
// call.  This entry point serves them: it runs the same span-aggregate, scan
// and read-out kernels as la_forward_noncausal, but takes its scratch (the
// per-span states and the head totals) from g_noalloc_scratch, and it calls
// no cudaMalloc, cudaFree or other allocating routine.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "linattn.h"
#include "noncausal_ffma.cuh"

namespace la {
namespace {

// Scratch shared by every call on a device; it keeps the last call's contents.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
struct NoAllocDevice {
    std::atomic<bool> ready{false};  // set (release) once the fields below are filled
    int num_sms = 0;
    float* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
NoAllocDevice g_na[kMaxDev];
std::mutex g_na_mu;

la_status na_fail(la_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    set_error_message(buf);
    return s;
}

// Once per device, with that device current: the SM count and the device
// address of the scratch array (in host code the array's name is only a
// host-side stand-in, never a usable device address).
la_status na_setup(NoAllocDevice** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return na_fail(LA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDev) return na_fail(LA_ERR_CUDA, "device ordinal %d out of range", dev);
    NoAllocDevice& d = g_na[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_na_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return na_fail(LA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
                return na_fail(LA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
            d.num_sms = sms;
            d.scratch = static_cast<float*>(p);
            d.ready.store(true, std::memory_order_release);
        }
    }
    *out = &d;
    return LA_OK;
}

template <typename T, int D, int M>
la_status run(const NoAllocDevice& dev, cudaStream_t st, const void* Qv, const void* Kv,
              const void* Vv, void* Ov, int BH, int N) {
    using namespace ffma;
    using C = Cfg<D, M>;
    const T* Q = static_cast<const T*>(Qv);
    const T* K = static_cast<const T*>(Kv);
    const T* V = static_cast<const T*>(Vv);
    T* O = static_cast<T*>(Ov);
    int spans, span_len;
    choose_spans(BH, N, C::L, dev.num_sms, &spans, &span_len);
    // Fewer spans when the span states would not fit (spans + 1 states per head).
    const size_t head_bytes = sizeof(float) * (size_t)C::W;
    const size_t cap_states = kNoAllocScratchBytes / head_bytes;
    if (cap_states < 2 * (size_t)BH)
        return na_fail(LA_ERR_INVALID_ARG,
                       "la_forward_noncausal_noalloc: B*H=%d needs %zu bytes of scratch at D=%d "
                       "M=%d, the fixed scratch holds %zu",
                       BH, 2 * (size_t)BH * head_bytes, D, M, kNoAllocScratchBytes);
    const int max_spans = (int)(cap_states / (size_t)BH) - 1;
    if (spans > max_spans) {
        const int chunks = (N + C::L - 1) / C::L;
        const int per = (chunks + max_spans - 1) / max_spans;
        span_len = per * C::L;
        spans = (N + span_len - 1) / span_len;
    }
    float* agg = dev.scratch;
    float* totals = dev.scratch + (size_t)BH * spans * C::W;
    cudaError_t e;
    if ((e = allow_smem(span_aggregate_kernel<T, D, M>, Smem<D, M>::agg)) != cudaSuccess)
        return na_fail(LA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    span_aggregate_kernel<T, D, M><<<dim3(BH, spans), kThreads, Smem<D, M>::agg, st>>>(
        K, V, agg, N, spans, span_len);
    const size_t n = (size_t)BH * C::W;
    span_scan_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(agg, nullptr, nullptr, totals,
                                                                 BH, spans, D, M, 0);
    const size_t smem = sizeof(float) * (D * C::MP + D + C::L * C::DP + C::L);
    if ((e = allow_smem(noncausal_out_kernel<T, D, M>, smem)) != cudaSuccess)
        return na_fail(LA_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    noncausal_out_kernel<T, D, M><<<dim3(BH, spans), kThreads, smem, st>>>(Q, O, totals, N,
                                                                          span_len);
    note_launch(3);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return na_fail(LA_ERR_CUDA, "la_forward_noncausal_noalloc: %s", cudaGetErrorString(e));
    return LA_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool head_ok(int x) { return x == 32 || x == 64 || x == 128; }

}  // namespace
}  // namespace la

extern "C" la_status la_forward_noncausal_noalloc(const void* Q, const void* K, const void* V,
                                                  void* Out, int B, int H, int N, int D, int M,
                                                  la_dtype dtype, void* stream) {
    using namespace la;
    if (B < 0 || H < 0 || N < 0)
        return na_fail(LA_ERR_INVALID_ARG, "la_forward_noncausal_noalloc: negative size");
    if (dtype != LA_DTYPE_F32 && dtype != LA_DTYPE_BF16)
        return na_fail(LA_ERR_UNSUPPORTED, "la_forward_noncausal_noalloc: unknown dtype %d", (int)dtype);
    if (!head_ok(D) || !head_ok(M))
        return na_fail(LA_ERR_UNSUPPORTED,
                       "la_forward_noncausal_noalloc: D=%d M=%d, supported head sizes are 32, 64, 128",
                       D, M);
    const unsigned long long bh = (unsigned long long)B * H;
    if (bh >= (1ull << 31) || bh * N * (unsigned long long)(D > M ? D : M) >= (1ull << 40))
        return na_fail(LA_ERR_INVALID_ARG, "la_forward_noncausal_noalloc: tensor too large");
    if (bh * N == 0) return LA_OK;
    const void* ptrs[] = {Q, K, V, Out};
    const char* names[] = {"Q", "K", "V", "Out"};
    for (int i = 0; i < 4; ++i) {
        if (!ptrs[i]) return na_fail(LA_ERR_INVALID_ARG, "la_forward_noncausal_noalloc: %s is NULL", names[i]);
        if (!al16(ptrs[i]))
            return na_fail(LA_ERR_INVALID_ARG, "la_forward_noncausal_noalloc: %s is not 16-byte aligned",
                           names[i]);
    }
    NoAllocDevice* dev = nullptr;
    la_status s = na_setup(&dev);
    if (s != LA_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
#define LA_NA_CASE(T, d, m) \
    if (D == d && M == m) return run<T, d, m>(*dev, st, Q, K, V, Out, (int)bh, N);
#define LA_NA_T(T)                                                                   \
    LA_NA_CASE(T, 32, 32) LA_NA_CASE(T, 32, 64) LA_NA_CASE(T, 32, 128)               \
    LA_NA_CASE(T, 64, 32) LA_NA_CASE(T, 64, 64) LA_NA_CASE(T, 64, 128)               \
    LA_NA_CASE(T, 128, 32) LA_NA_CASE(T, 128, 64) LA_NA_CASE(T, 128, 128)
    if (dtype == LA_DTYPE_F32) {
        LA_NA_T(float)
    } else {
        LA_NA_T(__nv_bfloat16)
    }
    return na_fail(LA_ERR_UNSUPPORTED, "la_forward_noncausal_noalloc: unsupported shape");
}
