/*
 * linattn.h -- C ABI of the GB300 (sm_103a) kernelized linear-attention library.
 *
 * The method ("Transformers are RNNs", as explained on wkq9411.github.io,
 * "【论文解读】Transformers are RNNs"): with phi(x) = elu(x) + 1 (section
 * 特征映射, eq. elu, alpha = 1),
 *
 *     V'_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i,                       (eq. output)
 *     S_i  = sum_{j<=i} phi(K_j) V_j^T,   Z_i = sum_{j<=i} phi(K_j)   (section 三)
 *
 * in the causal case (diagonal included, eq. mask) and with full sums in the
 * non-causal case (section 二, eq. linear).  No scaling is applied to Q or K.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Tensors are contiguous, row-major, in DEVICE memory of the current CUDA
 *   device: Q, K are [B][H][N][D]; V, Out, dOut are [B][H][N][M]; states S are
 *   [B][H][D][M] and Z are [B][H][D], always fp32.  Every non-empty tensor
 *   pointer must be 16-byte aligned.
 * - dtype: LA_DTYPE_F32 (fp32 storage) or LA_DTYPE_BF16 (bf16 storage).
 *   Outputs have the input dtype, except decode `out` and all states (fp32).
 *   All accumulation is fp32.
 * - Supported head sizes: D, M in {32, 64, 128}.  B, H, N >= 0; a call with
 *   B*H*N == 0 does no work and succeeds.  B*H*N*max(D,M) < 2^40.
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *   asynchronous on that stream; arguments are validated on the host before
 *   anything is enqueued, and an invalid call enqueues nothing.
 * - Ownership: the caller owns every buffer it passes.  The library never
 *   frees caller memory.  Per-call scratch (span states, gradient rows) is
 *   taken stream-ordered from a library-owned CUDA memory pool of the current
 *   device and given back on the same stream; la_workspace_bytes gives its
 *   size for each call.
 * - Errors: a status code; no exception or abort crosses the ABI.  On error,
 *   la_last_error_message() gives a one-line reason (per host thread).
 *
 * Library scratch is stream-ordered, so calls on different streams may run
 * concurrently.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, overflow */
    LA_ERR_UNSUPPORTED = 2, /* D or M not in {32, 64, 128}, unknown dtype */
    LA_ERR_CUDA = 3,        /* a CUDA runtime call failed (message has details) */
    LA_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (see la_check_device_status) */
} la_status;

typedef enum { LA_DTYPE_F32 = 0, LA_DTYPE_BF16 = 1 } la_dtype;

/*
 * Causal forward V' = phi(Q) S_i / phi(Q) Z_i ("Transformers are RNNs",
 * section 三, eq. mask and eq. output).
 *   Q, K    [B][H][N][D] dtype          (read)
 *   V       [B][H][N][M] dtype          (read)
 *   Out     [B][H][N][M] dtype          (written)
 *   S_init  [B][H][D][M] fp32, nullable (read)  state before token 0 (0 if NULL)
 *   Z_init  [B][H][D]    fp32, nullable (read)  must be NULL iff S_init is NULL
 *   S_final [B][H][D][M] fp32, nullable (written) state after token N-1
 *   Z_final [B][H][D]    fp32, nullable (written) must be NULL iff S_final is NULL
 *   Den     [B][H][N]    fp32, nullable (written) the normaliser phi(Q_i).Z_i
 *           of every token (the denominator of eq. output), for the backward
 *   Ckpt    fp32, nullable (written) la_causal_ckpt_floats(B, H, N, D, M)
 *           words: the state (S_i, Z_i) of every head before every 1024th
 *           token, for the backward (written by the bf16 D = M = 64 path;
 *           the other paths leave it untouched)
 * With S_init/Z_init a sequence can be processed in pieces; S_final/Z_final
 * hand a prefill's state to la_decode_step (section 三（二）: the state phi(K)V^T
 * is kept as an internal RNN state).  Out, Den and Ckpt may not alias any input.
 */
la_status la_forward_causal(const void* Q, const void* K, const void* V, void* Out,
                            int B, int H, int N, int D, int M, la_dtype dtype,
                            const float* S_init, const float* Z_init,
                            float* S_final, float* Z_final, float* Den, float* Ckpt,
                            void* stream);

/*
 * Size in fp32 words of the optional state checkpoints of la_forward_causal /
 * la_backward_causal: B * H * ceil(ceil(N / 128) / 8) * (D * M + D), or 0 for
 * non-positive sizes.  Pure arithmetic; no device call.
 */
size_t la_causal_ckpt_floats(int B, int H, int N, int D, int M);

/*
 * Causal backward of L(Out) given dOut = dL/dOut: the numerator gradients of
 * section 三（一）4 (eqs. gq-gv: a prefix state for phi(Q), a suffix state for
 * phi(K) and V), the denominator by the quotient rule, then the chain rule
 * through phi.
 *   Q, K [B][H][N][D]; V, dOut [B][H][N][M] dtype        (read)
 *   Out  [B][H][N][M] dtype, nullable                    (read) the forward's
 *        output; when NULL it is recomputed.
 *   Den  [B][H][N] fp32, nullable                        (read) the forward's
 *        normaliser per token (la_forward_causal's Den, from the same inputs);
 *        the bf16 D = M = 64 path then skips recomputing it, the other paths
 *        ignore it.  The results agree within the bf16 tolerance either way.
 *   Ckpt nullable (read) la_forward_causal's checkpoints from the same inputs
 *        and no S_init; the bf16 D = M = 64 path then starts each part of a
 *        sequence from the nearest one instead of re-reading K and V from the
 *        head's start; the other paths ignore it.
 *   dQ, dK [B][H][N][D]; dV [B][H][N][M] dtype           (written)
 * Outputs may not alias inputs or each other.
 */
la_status la_backward_causal(const void* Q, const void* K, const void* V, const void* Out,
                             const void* dOut, void* dQ, void* dK, void* dV,
                             int B, int H, int N, int D, int M, la_dtype dtype,
                             const float* Den, const float* Ckpt, void* stream);

/*
 * Non-causal forward V' = phi(Q)(phi(K)^T V) / phi(Q) sum_j phi(K_j)
 * ("Transformers are RNNs", section 二, eq. linear and the matrix form
 * (phi(Q)phi(K)^T)V = phi(Q)(phi(K)^T V)).
 *   Q, K [B][H][N][D]; V [B][H][N][M] dtype (read);  Out [B][H][N][M] dtype (written).
 * The call's kernels run in `stream` after the caller's earlier work there.
 * On the fp32 D = M = 64 path the read-out kernel is launched as a
 * programmatic dependent of the state kernel (it starts under that kernel's
 * tail and waits for its partials itself); the chain stays inside the call,
 * and a CUDA graph that captures the call keeps it.
 */
la_status la_forward_noncausal(const void* Q, const void* K, const void* V, void* Out,
                               int B, int H, int N, int D, int M, la_dtype dtype,
                               void* stream);

/*
 * Non-causal backward: the gradient of L(Out) given dOut = dL/dOut for
 * la_forward_noncausal's output.  The numerator gradients of "Transformers
 * are RNNs" section 三（一）4 (eqs. gq-gv) with the prefix state of phi(Q) and
 * the suffix state of phi(K) and V both summed over every token (the
 * unmasked sums of section 二, eq. linear), the denominator by the quotient
 * rule, then the chain rule through phi:
 *   gn_i = dOut_i / den_i, gd_i = -(dOut_i . Out_i) / den_i, den_i = phi(Q_i).Z
 *   dphi(Q_i) = S gn_i + Z gd_i;  R = sum_i phi(Q_i) gn_i^T, r = sum_i phi(Q_i) gd_i
 *   dphi(K_j) = R V_j + r;  dV_j = R^T phi(K_j)
 *   Q, K [B][H][N][D]; V, dOut [B][H][N][M] dtype   (read)
 *   Out  [B][H][N][M] dtype, nullable               (read) the forward's output;
 *        recomputed when NULL
 *   dQ, dK [B][H][N][D]; dV [B][H][N][M] dtype      (written)
 * Outputs may not alias inputs or each other.  On the fp32 D = M = 64 path
 * the call's three kernels are chained by programmatic dependent launch, as
 * in la_forward_noncausal; ordering with the caller's work is unchanged.
 */
la_status la_backward_noncausal(const void* Q, const void* K, const void* V, const void* Out,
                                const void* dOut, void* dQ, void* dK, void* dV,
                                int B, int H, int N, int D, int M, la_dtype dtype, void* stream);

/*
 * One recurrent decode step for B*H independent heads ("Transformers are
 * RNNs" section 四, the RNN form; "Transformer与RNN的深层联结" section 2,
 * RNN-mode inference): first S += phi(k) v^T and Z += phi(k), then
 * out = phi(q)^T S / phi(q)^T Z.
 *   q, k [B][H][D]; v [B][H][M] dtype     (read)
 *   S [B][H][D][M], Z [B][H][D] fp32      (read and updated in place)
 *   out [B][H][M] fp32                    (written)
 * The caller owns S and Z (a session's state can be saved, restored or moved
 * by copying them).  out may not alias S, Z or the inputs.
 */
la_status la_decode_step(const void* q, const void* k, const void* v, float* S, float* Z,
                         float* out, int B, int H, int D, int M, la_dtype dtype, void* stream);

/*
 * Attention with the degree-2 polynomial similarity sim(q, k) = (q^T k)^2 in
 * its linear form ("【论文解读】Transformers are RNNs", section 二 (3): the
 * explicit feature map phi(x) = (x_a x_b), C = D^2 features, cost O(N D^2 M)):
 *     V'_i = phi(Q_i)^T S / phi(Q_i)^T Z,  S = sum_j phi(K_j) V_j^T,  Z = sum_j phi(K_j)
 * over j <= i when causal != 0 (section 三), else over all j.  Raw Q and K
 * (no elu).  Q, K [B][H][N][D]; V [B][H][N][M] dtype (read); Out [B][H][N][M]
 * dtype (written).  Built for D = 32 and M in {32, 64} (LA_ERR_UNSUPPORTED
 * otherwise).  A row whose query is orthogonal to every key it sees has a zero
 * denominator and no defined output.
 */
la_status la_forward_poly2(const void* Q, const void* K, const void* V, void* Out, int B, int H,
                           int N, int D, int M, la_dtype dtype, int causal, void* stream);

/*
 * Linear attention with decay ("retention"), as "Transformer and Variants"
 * (by-xin.github.io) writes it: section 1.3.2 (linear attention as an RNN
 * without the reflection term, no softmax and no normaliser) and section
 * 1.3.4 (RetNet: a decay gamma per head; gated retention: a decay gamma_t per
 * token), with the state in the S = sum k v^T convention (the page's H
 * transposed):
 *     S_t = gamma_t S_{t-1} + k_t v_t^T,   Out_t = S_t^T q_t
 * Raw Q and K (no feature map).
 *   Q, K [B][H][N][D]; V [B][H][N][M] dtype (read);  Out [B][H][N][M] dtype (written)
 *   gamma_head [H] fp32, nullable: RetNet's decay of each head
 *   gates      [B][H][N] fp32, nullable: gated retention's decay of every token
 *              (the page's sigmoid(W_gamma x_t), computed by the caller)
 *   neither: decay 1 (the unnormalised form); both: LA_ERR_INVALID_ARG.
 *   Decays lie in (0, 1]; one below 2^-64 acts as 2^-64.
 *   S_init [B][H][D][M] fp32, nullable (read): state before token 0 (0 if NULL)
 *   S_final [B][H][D][M] fp32, nullable (written): state after token N-1
 */
la_status la_forward_retention(const void* Q, const void* K, const void* V, void* Out, int B,
                               int H, int N, int D, int M, la_dtype dtype, const float* gamma_head,
                               const float* gates, const float* S_init, float* S_final,
                               void* stream);

/*
 * One retention decode step for B*H heads: S = gamma S + k v^T, then
 * out = S^T q ("Transformer and Variants" section 1.3.4, RNN form).
 *   q, k [B][H][D]; v [B][H][M] dtype      (read)
 *   gamma_head [H] fp32, nullable; gate [B][H] fp32, nullable (this step's
 *   decay of each head); neither: decay 1
 *   S [B][H][D][M] fp32                    (read and updated in place)
 *   out [B][H][M] fp32                     (written)
 */
la_status la_retention_decode_step(const void* q, const void* k, const void* v,
                                   const float* gamma_head, const float* gate, float* S, float* out,
                                   int B, int H, int D, int M, la_dtype dtype, void* stream);

/*
 * One decode step of standard softmax attention with a KV cache, the baseline
 * the recurrent step is measured against ("Transformer与RNN的深层联结",
 * section 2, standard Transformer inference: the step's k, v are appended to
 * the cache, then out = softmax(q K^T / sqrt(D)) V over every cached position;
 * the scaled dot product of "Transformers are RNNs", section 一, eq. softmax).
 * Its cost grows with the cache; la_decode_step's does not.
 *   q, k [B][H][D]; v [B][H][M] dtype               (read)
 *   K_cache [B][H][T_max][D], V_cache [B][H][T_max][M] dtype
 *           rows 0..T-1 read; row T written with k, v
 *   T       positions already cached, 0 <= T < T_max (same for every head)
 *   out     [B][H][M] fp32                          (written)
 * Needs D == M (in {32, 64, 128}); LA_ERR_UNSUPPORTED otherwise.  Scratch:
 * la_workspace_bytes("la_softmax_decode_step", B, H, T, D, M, ...).
 */
la_status la_softmax_decode_step(const void* q, const void* k, const void* v, void* K_cache,
                                 void* V_cache, int T, int T_max, float* out, int B, int H, int D,
                                 int M, la_dtype dtype, void* stream);

/*
 * la_forward_noncausal with no device allocation.  The paper has no
 * counterpart: this is a service for callers that may not allocate device
 * memory inside an op -- a host framework that plans all device memory in
 * advance and gives the op only its inputs and outputs, a plugin runtime that
 * forbids allocation, or a latency-critical loop that cannot pay for an
 * allocator call.  Arguments, layouts and results are those of
 * la_forward_noncausal (up to the order of floating-point summation).
 * Its scratch is one fixed 16 MiB file-scope device array per device.  With
 * CUDA's default lazy module loading the array is committed on a device by
 * the first call there (its address lookup loads the library's device code),
 * and it stays until the process exits, so a caller that plans device memory
 * should make that first call before planning; later calls make no
 * cudaMalloc, cudaFree or other allocating call.  Limit: 2 * B * H * (D*M + D) * 4 bytes must fit in 16 MiB (B*H <= 127
 * at D = M = 128, <= 504 at D = M = 64); larger calls return
 * LA_ERR_INVALID_ARG with the sizes in the message.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current, so make the first call on each device before any stream
 * capture.  Every call on a device shares the one array and leaves its
 * contents behind; calls whose work overlaps on the GPU (e.g. on two streams)
 * race on it and must be serialised by the caller.
 */
la_status la_forward_noncausal_noalloc(const void* Q, const void* K, const void* V, void* Out,
                                       int B, int H, int N, int D, int M, la_dtype dtype,
                                       void* stream);

/*
 * Scratch of one call, for callers that plan device memory.  The pages'
 * interface keeps the state S, Z (and for the backward the suffix state)
 * inside the operation ("Overview of Linear Attention", Algorithm forward /
 * backward; "Transformer与RNN的深层联结" section 2, the decode loop on
 * state_s, state_z); this library keeps the per-range states, flags and
 * gradient rows that its parallel split needs in a library-owned pool, and
 * this function says how many bytes of it one call holds at its peak.
 *   op       the entry point's name: "la_forward_causal", "la_backward_causal",
 *            "la_forward_noncausal", "la_backward_noncausal", "la_decode_step" (0),
 *            "la_softmax_decode_step" (N = the cache position T),
 *            "la_forward_retention", "la_retention_decode_step" (0),
 *            "la_forward_poly2" or
 *            "la_forward_noncausal_noalloc" (0: it uses its fixed array)
 *   B..M, dtype  the call's sizes and dtype (N is ignored for decode)
 *   saved    for "la_backward_causal": an OR of LA_SAVED_OUT, LA_SAVED_DEN and
 *            LA_SAVED_CKPT for the optional inputs the call will pass
 *            (Out == NULL makes the call recompute the forward, which needs more)
 *   num_sms  SM count of the device the call will run on; <= 0 queries the
 *            current device (the only device call this function makes)
 * Returns the bytes (0 when the call takes no scratch), or SIZE_MAX for an
 * unknown op, unsupported sizes or a failed device query, with the reason in
 * la_last_error_message().  Pure arithmetic when num_sms > 0.
 */
#define LA_SAVED_OUT 1u
#define LA_SAVED_DEN 2u
#define LA_SAVED_CKPT 4u
size_t la_workspace_bytes(const char* op, int B, int H, int N, int D, int M, la_dtype dtype,
                          unsigned saved, int num_sms);

/*
 * Highest number of bytes of the library's scratch pool on the current device
 * held at once since the pool was created or last reset; reset != 0 then sets
 * it back to zero (to the bytes held now).  For checking la_workspace_bytes
 * against what calls actually take.  SIZE_MAX if a CUDA call failed.
 */
size_t la_scratch_peak_bytes(int reset);

/*
 * Test hook for the failure path of the real kernels, off unless called: the
 * next library call on this process that launches the tensor-core causal
 * forward or backward has unit `unit` of its work split skip its look-back
 * publication (the flag that later units of the same head wait for), and
 * gives every look-back wait of that launch `spin_limit` polls (about 0.3 us
 * each) instead of the default.  The units waiting on the missing flag give
 * up, set the look-back bit (0x2) in the device error word, drain their copies
 * in flight, free their tensor memory and end, so the call returns without a
 * hang; its outputs are then undefined, and la_check_device_status reports
 * LA_ERR_TIMEOUT.  The setting is consumed by that one call.  LA_ERR_INVALID_ARG
 * for unit < 0 or spin_limit == 0.
 */
la_status la_debug_withhold_publication(int unit, unsigned spin_limit);

/* Synchronises `stream`, then reads and clears the current device's error
 * word set by bounded device-side waits.  LA_ERR_TIMEOUT if one gave up since
 * the last check, LA_ERR_CUDA if the stream reported an error, else LA_OK. */
la_status la_check_device_status(void* stream);

/* Launches one block whose two bounded device waits cannot be met -- an
 * mbarrier phase that nothing completes and a flag that nothing sets, each
 * given up after a few thousand polls (milliseconds) -- so that both set their
 * bits in the current device's error word, the word and bits the library's
 * kernels set when a copy, a product or a look-back flag never arrives.  For
 * testing that failure path: the next la_check_device_status(stream) reports
 * LA_ERR_TIMEOUT (code 0x3) and clears the word, and the device stays usable.
 * Asynchronous on `stream` (a cudaStream_t, NULL for the default stream);
 * LA_OK once launched, LA_ERR_CUDA if the launch failed. */
la_status la_selftest_expired_waits(void* stream);

/* Static text of a status code. */
const char* la_status_string(la_status status);

/* One-line reason for the last non-LA_OK status returned on this host thread. */
const char* la_last_error_message(void);

/* Number of kernels this library has launched in this process. */
uint64_t la_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* LINATTN_H */
