// la_launch.h -- host-side launchers behind the C ABI (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace la {

// Everything a launcher needs from the device it runs on.
struct LaunchCtx {
    cudaStream_t stream;
    int num_sms;
    cudaMemPool_t pool;          // library-owned pool for stream-ordered scratch
    unsigned int* status_word;   // device error word for bounded waits
    // test hook (la_debug_withhold_publication): the unit whose look-back flag the next
    // tensor-core causal launch leaves unset (-1: none), and its flag-poll limit (0: default)
    int withhold_unit;
    unsigned spin_limit;
};

// Counts one kernel launch (la_kernel_launch_count).
void note_launch(int n = 1);

// Sets the text returned by la_last_error_message() on this host thread.
void set_error_message(const char* msg);

// Optional checkpoints kept by the causal forward for the backward: the fp32
// state [S | Z] (D*M + D words) of every head before every kCkptChunks-th chunk
// of 128 tokens, laid out [BH][ceil(chunks / kCkptChunks)][D*M + D]; slot 0
// (the zero state) is never written or read.
constexpr int kCkptChunks = 8;

// Scratch bytes the tensor-core launchers take from the pool for one call
// (what la_workspace_bytes reports; the launchers allocate exactly these).
size_t causal_forward_tc_scratch(int D, int BH, int N, int num_sms);
size_t causal_backward_tc64_scratch(int BH, int N, int num_sms, bool out_given, bool den_given,
                                    bool ckpt_given);
size_t noncausal_forward_tc_f32_scratch(int BH, int N, int num_sms);

// Stream-ordered scratch from the library pool.  Returns cudaSuccess or the error.
cudaError_t scratch_alloc(const LaunchCtx& c, void** p, size_t bytes);
// One block whose bounded waits expire and set their bits in c.status_word.
cudaError_t selftest_expired_waits(const LaunchCtx& c);
void scratch_free(const LaunchCtx& c, void* p);

// Each launcher returns cudaSuccess or the first CUDA error it met.
template <typename T, int D, int M>
cudaError_t causal_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O, int BH,
                           int N, const float* S_init, const float* Z_init, float* S_final,
                           float* Z_final, float* Den);

// Tensor-core causal forward for bf16 storage with D = M in {64, 128}.
template <int D, int M>
cudaError_t causal_forward_tc(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                              const __nv_bfloat16* V, __nv_bfloat16* O, int BH, int N,
                              const float* S_init, const float* Z_init, float* S_final,
                              float* Z_final, float* Den, float* Ckpt);

// Tensor-core retention forward (decay, no normaliser) for bf16 storage with D = M in {64, 128}.
template <int D, int M>
cudaError_t retention_forward_tc(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                 const __nv_bfloat16* V, __nv_bfloat16* O, const float* gamma_head,
                                 const float* gates, int BH, int H, int N, const float* S_init,
                                 float* S_final);
size_t retention_forward_tc_scratch(int D, int BH, int N, int num_sms);

// Tensor-core causal backward for bf16 storage with D = M = 64; Den (the
// forward's normaliser per token) and Ckpt (its state checkpoints) may be null.
cudaError_t causal_backward_tc64(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                                 const __nv_bfloat16* V, const __nv_bfloat16* O,
                                 const __nv_bfloat16* G, __nv_bfloat16* dQ, __nv_bfloat16* dK,
                                 __nv_bfloat16* dV, int BH, int N, const float* Den,
                                 const float* Ckpt);

template <typename T, int D, int M>
cudaError_t causal_backward(const LaunchCtx& c, const T* Q, const T* K, const T* V, const T* O,
                            const T* G, T* dQ, T* dK, T* dV, int BH, int N);

// Tensor-core non-causal forward for fp32 storage with D = M = 64 (fp32
// operands split into two bf16 terms).
cudaError_t noncausal_forward_tc_f32(const LaunchCtx& c, const float* Q, const float* K,
                                     const float* V, float* O, int BH, int N);

template <typename T, int D, int M>
cudaError_t noncausal_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O,
                              int BH, int N);

// Tensor-core non-causal backward for fp32 storage with D = M = 64 (O nullable).
cudaError_t noncausal_backward_tc_f32(const LaunchCtx& c, const float* Q, const float* K,
                                      const float* V, const float* O, const float* G, float* dQ,
                                      float* dK, float* dV, int BH, int N);
size_t noncausal_backward_tc_f32_scratch(int BH, int N, int num_sms);

template <typename T, int D, int M>
cudaError_t noncausal_backward(const LaunchCtx& c, const T* Q, const T* K, const T* V, const T* O,
                               const T* G, T* dQ, T* dK, T* dV, int BH, int N);

// Softmax attention decode step with a KV cache (M = D): appends k, v at
// position T_len of the caches, then attends over positions 0..T_len.
template <typename T, int D>
cudaError_t softmax_decode_step(const LaunchCtx& c, const T* q, const T* k, const T* v, T* Kc,
                                T* Vc, int T_len, int T_max, float* out, int BH);

// Retention (decayed, unnormalised linear attention) forward on the CUDA cores:
// gamma_head [H] or gates [BH][N] (per token) or neither (decay 1).
template <typename T, int D, int M>
cudaError_t retention_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O,
                              const float* gamma_head, const float* gates, int BH, int H, int N,
                              const float* S_init, float* S_final);

// One retention decode step: S = gamma S + k v^T, out = S^T q.
template <typename T, int D, int M>
cudaError_t retention_step(const LaunchCtx& c, const T* q, const T* k, const T* v,
                           const float* gamma_head, const float* gate, float* S, float* out, int BH,
                           int H);

// Attention with the degree-2 polynomial similarity (q . k)^2 through its
// explicit feature map, D = 32, causal or over all tokens.
template <typename T, int M>
cudaError_t poly2_forward(const LaunchCtx& c, const T* Q, const T* K, const T* V, T* O, int BH,
                          int N, bool causal);

// The same on the tensor core for bf16 storage and M = 64 (D^2 = 1024 features).
cudaError_t poly2_forward_tc(const LaunchCtx& c, const __nv_bfloat16* Q, const __nv_bfloat16* K,
                             const __nv_bfloat16* V, __nv_bfloat16* O, int BH, int N, bool causal);

template <typename T, int D, int M>
cudaError_t decode_step(const LaunchCtx& c, const T* q, const T* k, const T* v, float* S,
                        float* Z, float* out, int BH);

}  // namespace la
