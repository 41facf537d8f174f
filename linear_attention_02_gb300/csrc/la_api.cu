// la_api.cu -- the C ABI declared in include/linattn.h: argument validation,
// per-device context (SM count, scratch pool, device error word) and dispatch
// to the kernels for each (dtype, D, M).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "la_launch.h"
#include "la_plan.h"
#include "linattn.h"

namespace la {

namespace {

std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_withhold_unit{-1};     // test hook, consumed by the next call
std::atomic<unsigned> g_spin_limit{0};
thread_local char g_msg[512] = "";

la_status fail(la_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

la_status cuda_fail(cudaError_t e, const char* where) {
    return fail(LA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceState {
    std::atomic<bool> ready{false};  // set (release) once the fields below are filled
    int num_sms = 0;
    cudaMemPool_t pool = nullptr;
    unsigned int* status_word = nullptr;
};
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

la_status get_ctx(cudaStream_t stream, LaunchCtx* ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(LA_ERR_CUDA, "device ordinal %d out of range", dev);
    DeviceState& d = g_dev[dev];
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (!d.ready.load(std::memory_order_relaxed)) {
            int sms = 0;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)))
                return cuda_fail(e, "cudaDeviceGetAttribute");
            cudaMemPoolProps props;
            memset(&props, 0, sizeof(props));
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cudaMemPool_t pool = nullptr;
            if ((e = cudaMemPoolCreate(&pool, &props))) return cuda_fail(e, "cudaMemPoolCreate");
            uint64_t keep = ~0ull;  // keep freed scratch in the pool between calls
            if ((e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep)))
                return cuda_fail(e, "cudaMemPoolSetAttribute");
            unsigned int* word = nullptr;
            if ((e = cudaMalloc(&word, 256))) return cuda_fail(e, "cudaMalloc(status word)");
            if ((e = cudaMemset(word, 0, 256))) return cuda_fail(e, "cudaMemset(status word)");
            d.num_sms = sms;
            d.pool = pool;
            d.status_word = word;
            d.ready.store(true, std::memory_order_release);
        }
    }
    ctx->stream = stream;
    ctx->withhold_unit = g_withhold_unit.exchange(-1);
    ctx->spin_limit = g_spin_limit.exchange(0u);
    ctx->num_sms = d.num_sms;
    ctx->pool = d.pool;
    ctx->status_word = d.status_word;
    return LA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool head_ok(int x) { return x == 32 || x == 64 || x == 128; }

// Common shape/pointer checks.  `ptrs` must be non-null and 16-byte aligned
// whenever the work is non-empty.
la_status check_common(const char* fn, int B, int H, int N, int D, int M, la_dtype dt,
                       const void* const* ptrs, const char* const* names, int nptr,
                       bool* empty) {
    if (B < 0 || H < 0 || N < 0)
        return fail(LA_ERR_INVALID_ARG, "%s: negative size B=%d H=%d N=%d", fn, B, H, N);
    if (dt != LA_DTYPE_F32 && dt != LA_DTYPE_BF16)
        return fail(LA_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dt);
    if (!head_ok(D) || !head_ok(M))
        return fail(LA_ERR_UNSUPPORTED, "%s: D=%d M=%d, supported head sizes are 32, 64, 128", fn,
                    D, M);
    const unsigned long long bhn = (unsigned long long)B * H * N;
    if (bhn * (unsigned long long)(D > M ? D : M) >= (1ull << 40))
        return fail(LA_ERR_INVALID_ARG, "%s: tensor too large", fn);
    if ((unsigned long long)B * H >= (1ull << 31))
        return fail(LA_ERR_INVALID_ARG, "%s: B*H too large", fn);
    *empty = bhn == 0;
    if (*empty) return LA_OK;
    for (int i = 0; i < nptr; ++i) {
        if (!ptrs[i]) return fail(LA_ERR_INVALID_ARG, "%s: %s is NULL", fn, names[i]);
        if (!aligned16(ptrs[i]))
            return fail(LA_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, names[i]);
    }
    return LA_OK;
}

la_status check_optional(const char* fn, const void* p, const char* name) {
    if (p && !aligned16(p)) return fail(LA_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, name);
    return LA_OK;
}

la_status finish(cudaError_t e, const char* fn) {
    if (e != cudaSuccess) return cuda_fail(e, fn);
    return LA_OK;
}

// Calls F::template run<T, D, M>(args...) for the runtime (dtype, D, M).
template <class F, class... A>
cudaError_t dispatch(la_dtype dt, int D, int M, A... a) {
#define LA_CASE_DM(T, d, m) \
    if (D == d && M == m) return F::template run<T, d, m>(a...);
#define LA_CASE_T(T)                                                                  \
    LA_CASE_DM(T, 32, 32) LA_CASE_DM(T, 32, 64) LA_CASE_DM(T, 32, 128)                \
    LA_CASE_DM(T, 64, 32) LA_CASE_DM(T, 64, 64) LA_CASE_DM(T, 64, 128)                \
    LA_CASE_DM(T, 128, 32) LA_CASE_DM(T, 128, 64) LA_CASE_DM(T, 128, 128)
    if (dt == LA_DTYPE_F32) {
        LA_CASE_T(float)
    } else {
        LA_CASE_T(__nv_bfloat16)
    }
#undef LA_CASE_T
#undef LA_CASE_DM
    return cudaErrorInvalidValue;
}

// bf16 with D = M in {64, 128} runs on the tensor cores; every other shape
// and fp32 storage runs the CUDA-core kernels.
template <typename T, int D, int M>
struct UseTensorCores {
    static constexpr bool value = false;
};
template <>
struct UseTensorCores<__nv_bfloat16, 64, 64> {
    static constexpr bool value = true;
};
template <>
struct UseTensorCores<__nv_bfloat16, 128, 128> {
    static constexpr bool value = true;
};

struct FwdCausal {
    template <typename T, int D, int M>
    static cudaError_t run(const LaunchCtx* c, const void* Q, const void* K, const void* V, void* O,
                           int BH, int N, const float* Si, const float* Zi, float* Sf, float* Zf,
                           float* Den, float* Ckpt) {
        if constexpr (UseTensorCores<T, D, M>::value)
            return causal_forward_tc<D, M>(*c, (const T*)Q, (const T*)K, (const T*)V, (T*)O, BH, N,
                                           Si, Zi, Sf, Zf, Den, Ckpt);
        else
            return causal_forward<T, D, M>(*c, (const T*)Q, (const T*)K, (const T*)V, (T*)O, BH, N,
                                           Si, Zi, Sf, Zf, Den);
    }
};
struct BwdCausal {
    template <typename T, int D, int M>
    static cudaError_t run(const LaunchCtx* c, const void* Q, const void* K, const void* V,
                           const void* O, const void* G, void* dQ, void* dK, void* dV, int BH, int N,
                           const float* Den, const float* Ckpt) {
        if constexpr (std::is_same<T, __nv_bfloat16>::value && D == 64 && M == 64)
            return causal_backward_tc64(*c, (const T*)Q, (const T*)K, (const T*)V, (const T*)O,
                                        (const T*)G, (T*)dQ, (T*)dK, (T*)dV, BH, N, Den, Ckpt);
        else
            return causal_backward<T, D, M>(*c, (const T*)Q, (const T*)K, (const T*)V,
                                            (const T*)O, (const T*)G, (T*)dQ, (T*)dK, (T*)dV, BH,
                                            N);
    }
};
struct FwdNoncausal {
    template <typename T, int D, int M>
    static cudaError_t run(const LaunchCtx* c, const void* Q, const void* K, const void* V, void* O,
                           int BH, int N) {
        if constexpr (std::is_same<T, float>::value && D == 64 && M == 64)
            return noncausal_forward_tc_f32(*c, (const T*)Q, (const T*)K, (const T*)V, (T*)O, BH, N);
        else
            return noncausal_forward<T, D, M>(*c, (const T*)Q, (const T*)K, (const T*)V, (T*)O, BH,
                                              N);
    }
};
struct BwdNoncausal {
    template <typename T, int D, int M>
    static cudaError_t run(const LaunchCtx* c, const void* Q, const void* K, const void* V,
                           const void* O, const void* G, void* dQ, void* dK, void* dV, int BH, int N) {
        if constexpr (std::is_same<T, float>::value && D == 64 && M == 64)
            return noncausal_backward_tc_f32(*c, (const T*)Q, (const T*)K, (const T*)V, (const T*)O,
                                             (const T*)G, (T*)dQ, (T*)dK, (T*)dV, BH, N);
        else
            return noncausal_backward<T, D, M>(*c, (const T*)Q, (const T*)K, (const T*)V, (const T*)O,
                                               (const T*)G, (T*)dQ, (T*)dK, (T*)dV, BH, N);
    }
};
struct FwdRetention {
    template <typename T, int D, int M>
    static cudaError_t run(const LaunchCtx* c, const void* Q, const void* K, const void* V, void* O,
                           const float* gh, const float* gt, int BH, int H, int N, const float* Si,
                           float* Sf) {
        if constexpr (UseTensorCores<T, D, M>::value)
            return retention_forward_tc<D, M>(*c, (const T*)Q, (const T*)K, (const T*)V, (T*)O, gh,
                                              gt, BH, H, N, Si, Sf);
        else
            return retention_forward<T, D, M>(*c, (const T*)Q, (const T*)K, (const T*)V, (T*)O, gh,
                                              gt, BH, H, N, Si, Sf);
    }
};
struct RetentionStep {
    template <typename T, int D, int M>
    static cudaError_t run(const LaunchCtx* c, const void* q, const void* k, const void* v,
                           const float* gh, const float* gt, float* S, float* out, int BH, int H) {
        return retention_step<T, D, M>(*c, (const T*)q, (const T*)k, (const T*)v, gh, gt, S, out, BH,
                                       H);
    }
};
struct Decode {
    template <typename T, int D, int M>
    static cudaError_t run(const LaunchCtx* c, const void* q, const void* k, const void* v,
                           float* S, float* Z, float* out, int BH) {
        return decode_step<T, D, M>(*c, (const T*)q, (const T*)k, (const T*)v, S, Z, out, BH);
    }
};

// Writes zeros (or the initial state) to S_final/Z_final for an N == 0 forward.
cudaError_t empty_forward_state(cudaStream_t st, size_t bh, int D, int M, const float* Si,
                                const float* Zi, float* Sf, float* Zf) {
    if (!Sf || bh == 0) return cudaSuccess;
    const size_t sb = bh * D * M * sizeof(float), zb = bh * D * sizeof(float);
    cudaError_t e;
    if (Si) {
        if ((e = cudaMemcpyAsync(Sf, Si, sb, cudaMemcpyDeviceToDevice, st))) return e;
        return cudaMemcpyAsync(Zf, Zi, zb, cudaMemcpyDeviceToDevice, st);
    }
    if ((e = cudaMemsetAsync(Sf, 0, sb, st))) return e;
    return cudaMemsetAsync(Zf, 0, zb, st);
}

}  // namespace

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

void set_error_message(const char* msg) { snprintf(g_msg, sizeof(g_msg), "%s", msg); }

cudaError_t scratch_alloc(const LaunchCtx& c, void** p, size_t bytes) {
    if (bytes == 0) bytes = 256;
    return cudaMallocFromPoolAsync(p, bytes, c.pool, c.stream);
}

void scratch_free(const LaunchCtx& c, void* p) {
    if (p) cudaFreeAsync(p, c.stream);
}

// Scratch bytes of one call, following the same dispatch as the entry points.
size_t workspace_for(const char* op, int BH, int N, int D, int M, la_dtype dt, unsigned saved,
                     int sms) {
    const bool bf16 = dt == LA_DTYPE_BF16;
    if (!strcmp(op, "la_forward_causal")) {
        if (bf16 && D == M && (D == 64 || D == 128)) return causal_forward_tc_scratch(D, BH, N, sms);
        return plan::ffma_causal_forward(BH, N, D, M, sms);
    }
    if (!strcmp(op, "la_backward_causal")) {
        if (bf16 && D == 64 && M == 64)
            return causal_backward_tc64_scratch(BH, N, sms, saved & LA_SAVED_OUT, saved & LA_SAVED_DEN,
                                                saved & LA_SAVED_CKPT);
        return plan::ffma_causal_backward(BH, N, D, M, sms);
    }
    if (!strcmp(op, "la_forward_noncausal")) {
        if (!bf16 && D == 64 && M == 64) return noncausal_forward_tc_f32_scratch(BH, N, sms);
        return plan::ffma_noncausal_forward(BH, N, D, M, sms);
    }
    if (!strcmp(op, "la_backward_noncausal"))
        return !bf16 && D == 64 && M == 64 ? noncausal_backward_tc_f32_scratch(BH, N, sms)
                                           : plan::ffma_noncausal_backward(BH, N, D, M, sms);
    if (!strcmp(op, "la_forward_poly2")) {
        if (D != 32 || (M != 32 && M != 64)) return SIZE_MAX;
        return bf16 && M == 64 ? plan::poly2_tc_scratch(BH, N) : plan::poly2_scratch(BH, N, M, sms);
    }
    if (!strcmp(op, "la_forward_retention"))
        return bf16 && D == M && (D == 64 || D == 128) ? retention_forward_tc_scratch(D, BH, N, sms)
                                                       : plan::ffma_retention_forward(BH, N, D, M, sms);
    if (!strcmp(op, "la_retention_decode_step")) return 0;
    if (!strcmp(op, "la_softmax_decode_step"))  // N is the cache position T: T + 1 positions
        return D == M ? plan::softmax_decode_scratch(BH, N + 1, D, sms) : SIZE_MAX;
    if (!strcmp(op, "la_decode_step") || !strcmp(op, "la_forward_noncausal_noalloc")) return 0;
    return SIZE_MAX;
}

}  // namespace la

using namespace la;

extern "C" {

size_t la_workspace_bytes(const char* op, int B, int H, int N, int D, int M, la_dtype dtype,
                          unsigned saved, int num_sms) {
    static const char* fn = "la_workspace_bytes";
    if (!op) return fail(LA_ERR_INVALID_ARG, "%s: op is NULL", fn), SIZE_MAX;
    if (B < 0 || H < 0 || N < 0)
        return fail(LA_ERR_INVALID_ARG, "%s: negative size B=%d H=%d N=%d", fn, B, H, N), SIZE_MAX;
    if (dtype != LA_DTYPE_F32 && dtype != LA_DTYPE_BF16)
        return fail(LA_ERR_UNSUPPORTED, "%s: unknown dtype %d", fn, (int)dtype), SIZE_MAX;
    if (!head_ok(D) || !head_ok(M))
        return fail(LA_ERR_UNSUPPORTED, "%s: D=%d M=%d, supported head sizes are 32, 64, 128", fn, D,
                    M),
               SIZE_MAX;
    if ((unsigned long long)B * H >= (1ull << 31))
        return fail(LA_ERR_INVALID_ARG, "%s: B*H too large", fn), SIZE_MAX;
    const int BH = B * H;
    if (workspace_for(op, 1, 1, D, M, dtype, saved, 1) == SIZE_MAX)
        return fail(LA_ERR_INVALID_ARG, "%s: unknown op \"%s\" or unsupported shape", fn, op), SIZE_MAX;
    if (!strcmp(op, "la_decode_step")) N = 1;
    const bool cache_op = !strcmp(op, "la_softmax_decode_step");  // N = T may be 0
    if (BH == 0 || (N == 0 && !cache_op)) return 0;
    if (num_sms <= 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, fn), SIZE_MAX;
    }
    return workspace_for(op, BH, N, D, M, dtype, saved, num_sms);
}

size_t la_scratch_peak_bytes(int reset) {
    static const char* fn = "la_scratch_peak_bytes";
    LaunchCtx ctx;
    if (get_ctx(nullptr, &ctx) != LA_OK) return SIZE_MAX;
    unsigned long long v = 0;
    cudaError_t e = cudaMemPoolGetAttribute(ctx.pool, cudaMemPoolAttrUsedMemHigh, &v);
    if (e != cudaSuccess) return cuda_fail(e, fn), SIZE_MAX;
    if (reset) {
        unsigned long long zero = 0;
        if ((e = cudaMemPoolSetAttribute(ctx.pool, cudaMemPoolAttrUsedMemHigh, &zero)) != cudaSuccess)
            return cuda_fail(e, fn), SIZE_MAX;
    }
    return (size_t)v;
}


la_status la_forward_causal(const void* Q, const void* K, const void* V, void* Out, int B, int H,
                            int N, int D, int M, la_dtype dtype, const float* S_init,
                            const float* Z_init, float* S_final, float* Z_final, float* Den,
                            float* Ckpt, void* stream) {
    static const char* fn = "la_forward_causal";
    const void* p[] = {Q, K, V, Out};
    const char* nm[] = {"Q", "K", "V", "Out"};
    bool empty = false;
    la_status s = check_common(fn, B, H, N, D, M, dtype, p, nm, 4, &empty);
    if (s != LA_OK) return s;
    if ((S_init == nullptr) != (Z_init == nullptr))
        return fail(LA_ERR_INVALID_ARG, "%s: S_init and Z_init must both be given or both NULL", fn);
    if ((S_final == nullptr) != (Z_final == nullptr))
        return fail(LA_ERR_INVALID_ARG, "%s: S_final and Z_final must both be given or both NULL", fn);
    if ((s = check_optional(fn, S_init, "S_init")) || (s = check_optional(fn, Z_init, "Z_init")) ||
        (s = check_optional(fn, S_final, "S_final")) || (s = check_optional(fn, Z_final, "Z_final")) ||
        (s = check_optional(fn, Den, "Den")) || (s = check_optional(fn, Ckpt, "Ckpt")))
        return s;
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    const size_t bh = (size_t)B * H;
    if (empty) return finish(empty_forward_state(ctx.stream, bh, D, M, S_init, Z_init, S_final, Z_final), fn);
    return finish(dispatch<FwdCausal>(dtype, D, M, &ctx, Q, K, V, Out, (int)bh, N, S_init, Z_init,
                                      S_final, Z_final, Den, Ckpt),
                  fn);
}

la_status la_backward_causal(const void* Q, const void* K, const void* V, const void* Out,
                             const void* dOut, void* dQ, void* dK, void* dV, int B, int H, int N,
                             int D, int M, la_dtype dtype, const float* Den, const float* Ckpt,
                             void* stream) {
    static const char* fn = "la_backward_causal";
    const void* p[] = {Q, K, V, dOut, dQ, dK, dV};
    const char* nm[] = {"Q", "K", "V", "dOut", "dQ", "dK", "dV"};
    bool empty = false;
    la_status s = check_common(fn, B, H, N, D, M, dtype, p, nm, 7, &empty);
    if (s != LA_OK) return s;
    if ((s = check_optional(fn, Out, "Out")) || (s = check_optional(fn, Den, "Den")) ||
        (s = check_optional(fn, Ckpt, "Ckpt")))
        return s;
    if (empty) return LA_OK;
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    return finish(dispatch<BwdCausal>(dtype, D, M, &ctx, Q, K, V, Out, dOut, dQ, dK, dV,
                                      (int)((size_t)B * H), N, Den, Ckpt),
                  fn);
}

size_t la_causal_ckpt_floats(int B, int H, int N, int D, int M) {
    if (B <= 0 || H <= 0 || N <= 0 || D <= 0 || M <= 0) return 0;
    const size_t chunks = ((size_t)N + 127) / 128;
    return (size_t)B * H * ((chunks + kCkptChunks - 1) / kCkptChunks) * ((size_t)D * M + D);
}

la_status la_forward_noncausal(const void* Q, const void* K, const void* V, void* Out, int B,
                               int H, int N, int D, int M, la_dtype dtype, void* stream) {
    static const char* fn = "la_forward_noncausal";
    const void* p[] = {Q, K, V, Out};
    const char* nm[] = {"Q", "K", "V", "Out"};
    bool empty = false;
    la_status s = check_common(fn, B, H, N, D, M, dtype, p, nm, 4, &empty);
    if (s != LA_OK || empty) return s;
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    return finish(dispatch<FwdNoncausal>(dtype, D, M, &ctx, Q, K, V, Out, (int)((size_t)B * H), N),
                  fn);
}

la_status la_backward_noncausal(const void* Q, const void* K, const void* V, const void* Out,
                                const void* dOut, void* dQ, void* dK, void* dV, int B, int H, int N,
                                int D, int M, la_dtype dtype, void* stream) {
    static const char* fn = "la_backward_noncausal";
    const void* p[] = {Q, K, V, dOut, dQ, dK, dV};
    const char* nm[] = {"Q", "K", "V", "dOut", "dQ", "dK", "dV"};
    bool empty = false;
    la_status s = check_common(fn, B, H, N, D, M, dtype, p, nm, 7, &empty);
    if (s != LA_OK) return s;
    if ((s = check_optional(fn, Out, "Out"))) return s;
    if (empty) return LA_OK;
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    return finish(dispatch<BwdNoncausal>(dtype, D, M, &ctx, Q, K, V, Out, dOut, dQ, dK, dV,
                                         (int)((size_t)B * H), N),
                  fn);
}

la_status la_decode_step(const void* q, const void* k, const void* v, float* S, float* Z,
                         float* out, int B, int H, int D, int M, la_dtype dtype, void* stream) {
    static const char* fn = "la_decode_step";
    const void* p[] = {q, k, v, S, Z, out};
    const char* nm[] = {"q", "k", "v", "S", "Z", "out"};
    bool empty = false;
    la_status s = check_common(fn, B, H, 1, D, M, dtype, p, nm, 6, &empty);
    if (s != LA_OK || empty) return s;
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    return finish(dispatch<Decode>(dtype, D, M, &ctx, q, k, v, S, Z, out, (int)((size_t)B * H)), fn);
}

la_status la_forward_retention(const void* Q, const void* K, const void* V, void* Out, int B,
                               int H, int N, int D, int M, la_dtype dtype, const float* gamma_head,
                               const float* gates, const float* S_init, float* S_final,
                               void* stream) {
    static const char* fn = "la_forward_retention";
    const void* p[] = {Q, K, V, Out};
    const char* nm[] = {"Q", "K", "V", "Out"};
    bool empty = false;
    la_status s = check_common(fn, B, H, N, D, M, dtype, p, nm, 4, &empty);
    if (s != LA_OK) return s;
    if (gamma_head && gates)
        return fail(LA_ERR_INVALID_ARG, "%s: give gamma_head or gates, not both", fn);
    if ((s = check_optional(fn, S_init, "S_init")) || (s = check_optional(fn, S_final, "S_final")))
        return s;
    if (((uintptr_t)gamma_head | (uintptr_t)gates) & 3u)
        return fail(LA_ERR_INVALID_ARG, "%s: gamma_head / gates not 4-byte aligned", fn);
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    const size_t bh = (size_t)B * H;
    if (empty) {
        if (!S_final || bh == 0) return LA_OK;
        const size_t sb = bh * D * M * sizeof(float);
        return finish(S_init ? cudaMemcpyAsync(S_final, S_init, sb, cudaMemcpyDeviceToDevice, ctx.stream)
                             : cudaMemsetAsync(S_final, 0, sb, ctx.stream),
                      fn);
    }
    return finish(dispatch<FwdRetention>(dtype, D, M, &ctx, Q, K, V, Out, gamma_head, gates, (int)bh,
                                         H, N, S_init, S_final),
                  fn);
}

la_status la_retention_decode_step(const void* q, const void* k, const void* v,
                                   const float* gamma_head, const float* gate, float* S, float* out,
                                   int B, int H, int D, int M, la_dtype dtype, void* stream) {
    static const char* fn = "la_retention_decode_step";
    const void* p[] = {q, k, v, S, out};
    const char* nm[] = {"q", "k", "v", "S", "out"};
    bool empty = false;
    la_status s = check_common(fn, B, H, 1, D, M, dtype, p, nm, 5, &empty);
    if (s != LA_OK || empty) return s;
    if (gamma_head && gate) return fail(LA_ERR_INVALID_ARG, "%s: give gamma_head or gate, not both", fn);
    if (((uintptr_t)gamma_head | (uintptr_t)gate) & 3u)
        return fail(LA_ERR_INVALID_ARG, "%s: gamma_head / gate not 4-byte aligned", fn);
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    return finish(dispatch<RetentionStep>(dtype, D, M, &ctx, q, k, v, gamma_head, gate, S, out,
                                          (int)((size_t)B * H), H),
                  fn);
}

la_status la_forward_poly2(const void* Q, const void* K, const void* V, void* Out, int B, int H,
                           int N, int D, int M, la_dtype dtype, int causal, void* stream) {
    static const char* fn = "la_forward_poly2";
    const void* p[] = {Q, K, V, Out};
    const char* nm[] = {"Q", "K", "V", "Out"};
    bool empty = false;
    la_status s = check_common(fn, B, H, N, D, M, dtype, p, nm, 4, &empty);
    if (s != LA_OK) return s;
    if (D != 32 || (M != 32 && M != 64))
        return fail(LA_ERR_UNSUPPORTED, "%s: D=%d M=%d, the degree-2 feature map is built for D = 32, "
                    "M in {32, 64}", fn, D, M);
    if (empty) return LA_OK;
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    const int BH = B * H;
    const bool c = causal != 0;
    cudaError_t e;
    if (dtype == LA_DTYPE_F32)
        e = M == 32 ? poly2_forward<float, 32>(ctx, (const float*)Q, (const float*)K, (const float*)V,
                                               (float*)Out, BH, N, c)
                    : poly2_forward<float, 64>(ctx, (const float*)Q, (const float*)K, (const float*)V,
                                               (float*)Out, BH, N, c);
    else
        e = M == 32 ? poly2_forward<__nv_bfloat16, 32>(ctx, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K,
                                                       (const __nv_bfloat16*)V, (__nv_bfloat16*)Out, BH, N, c)
                    : poly2_forward_tc(ctx, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K,
                                       (const __nv_bfloat16*)V, (__nv_bfloat16*)Out, BH, N, c);
    return finish(e, fn);
}

la_status la_softmax_decode_step(const void* q, const void* k, const void* v, void* K_cache,
                                 void* V_cache, int T, int T_max, float* out, int B, int H, int D,
                                 int M, la_dtype dtype, void* stream) {
    static const char* fn = "la_softmax_decode_step";
    const void* p[] = {q, k, v, K_cache, V_cache, out};
    const char* nm[] = {"q", "k", "v", "K_cache", "V_cache", "out"};
    bool empty = false;
    la_status s = check_common(fn, B, H, 1, D, M, dtype, p, nm, 6, &empty);
    if (s != LA_OK) return s;
    if (D != M)
        return fail(LA_ERR_UNSUPPORTED, "%s: D=%d M=%d, the KV-cache step needs D == M", fn, D, M);
    if (T < 0 || T >= T_max)
        return fail(LA_ERR_INVALID_ARG, "%s: cache position T=%d must satisfy 0 <= T < T_max=%d", fn,
                    T, T_max);
    if ((unsigned long long)B * H * T_max * D >= (1ull << 40))
        return fail(LA_ERR_INVALID_ARG, "%s: cache too large", fn);
    if (empty) return LA_OK;
    LaunchCtx ctx;
    if ((s = get_ctx((cudaStream_t)stream, &ctx)) != LA_OK) return s;
    const int BH = B * H;
    cudaError_t e = cudaErrorInvalidValue;
#define LA_SD_CASE(Ty, d)                                                                       \
    if (D == d)                                                                                 \
        e = softmax_decode_step<Ty, d>(ctx, (const Ty*)q, (const Ty*)k, (const Ty*)v, (Ty*)K_cache, \
                                       (Ty*)V_cache, T, T_max, out, BH);
    if (dtype == LA_DTYPE_F32) {
        LA_SD_CASE(float, 32) else LA_SD_CASE(float, 64) else LA_SD_CASE(float, 128)
    } else {
        LA_SD_CASE(__nv_bfloat16, 32) else LA_SD_CASE(__nv_bfloat16, 64) else LA_SD_CASE(__nv_bfloat16, 128)
    }
#undef LA_SD_CASE
    return finish(e, fn);
}

la_status la_selftest_expired_waits(void* stream) {
    LaunchCtx ctx;
    la_status s = get_ctx((cudaStream_t)stream, &ctx);
    if (s != LA_OK) return s;
    return finish(selftest_expired_waits(ctx), "la_selftest_expired_waits");
}

la_status la_debug_withhold_publication(int unit, unsigned spin_limit) {
    if (unit < 0 || spin_limit == 0)
        return fail(LA_ERR_INVALID_ARG, "la_debug_withhold_publication: unit %d, spin limit %u", unit,
                    spin_limit);
    g_spin_limit.store(spin_limit);
    g_withhold_unit.store(unit);
    return LA_OK;
}

la_status la_check_device_status(void* stream) {
    LaunchCtx ctx;
    la_status s = get_ctx((cudaStream_t)stream, &ctx);
    if (s != LA_OK) return s;
    cudaError_t e = cudaStreamSynchronize(ctx.stream);
    if (e != cudaSuccess) return cuda_fail(e, "la_check_device_status");
    unsigned int word = 0;
    if ((e = cudaMemcpy(&word, ctx.status_word, sizeof(word), cudaMemcpyDeviceToHost)))
        return cuda_fail(e, "la_check_device_status");
    if (word) {
        const unsigned int zero = 0;
        if ((e = cudaMemcpy(ctx.status_word, &zero, sizeof(zero), cudaMemcpyHostToDevice)))
            return cuda_fail(e, "la_check_device_status");
        return fail(LA_ERR_TIMEOUT, "a bounded device wait gave up (code 0x%x)", word);
    }
    return LA_OK;
}

const char* la_status_string(la_status status) {
    switch (status) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
        case LA_ERR_CUDA: return "LA_ERR_CUDA";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
    }
    return "LA_ERR_UNKNOWN";
}

const char* la_last_error_message(void) { return g_msg; }

uint64_t la_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
