// la_plan.h -- host-side work splits and scratch sizes of the launchers
// (internal).  Each launcher takes from the library pool exactly the bytes the
// matching function here returns, so la_workspace_bytes can report them
// without touching the device.
#pragma once

#include <stddef.h>

#include <algorithm>

namespace la {
namespace plan {

// State words of one head: S (D x M) followed by Z (D).
constexpr size_t state_words(int D, int M) { return static_cast<size_t>(D) * M + D; }

// Chunk length of the CUDA-core (FFMA) kernels.
constexpr int ffma_chunk(int D, int M) { return (D >= 128 || M >= 128) ? 32 : 64; }

constexpr size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Spans per head of the CUDA-core kernels: enough CTAs for about two per SM,
// whole chunks per span.
inline void ffma_spans(int BH, int N, int L, int num_sms, int* spans, int* span_len) {
    const int chunks = (N + L - 1) / L;
    int s = (2 * num_sms + BH - 1) / std::max(BH, 1);
    s = std::max(1, std::min(s, chunks));
    const int per = (chunks + s - 1) / s;
    *span_len = per * L;
    *spans = (N + *span_len - 1) / *span_len;
}

inline int ffma_span_count(int BH, int N, int D, int M, int num_sms) {
    int spans = 1, len = 0;
    ffma_spans(BH, N, ffma_chunk(D, M), num_sms, &spans, &len);
    return spans;
}

// CUDA-core causal forward: the span aggregates, only when a head has several spans.
inline size_t ffma_causal_forward(int BH, int N, int D, int M, int num_sms) {
    const int spans = ffma_span_count(BH, N, D, M, num_sms);
    return spans > 1 ? sizeof(float) * static_cast<size_t>(BH) * spans * state_words(D, M) : 0;
}

// CUDA-core causal backward: S and R span aggregates, gn (fp32) and gd rows.
inline size_t ffma_causal_backward(int BH, int N, int D, int M, int num_sms) {
    const int spans = ffma_span_count(BH, N, D, M, num_sms);
    const size_t agg = sizeof(float) * static_cast<size_t>(BH) * spans * state_words(D, M);
    return 2 * agg + sizeof(float) * static_cast<size_t>(BH) * N * M +
           sizeof(float) * static_cast<size_t>(BH) * N + 256;
}

// CUDA-core non-causal forward: span aggregates plus the head totals.
inline size_t ffma_noncausal_forward(int BH, int N, int D, int M, int num_sms) {
    const int spans = ffma_span_count(BH, N, D, M, num_sms);
    return sizeof(float) * (static_cast<size_t>(BH) * spans + BH) * state_words(D, M);
}

// CUDA-core non-causal backward: state partials and totals, (R | r) partials and totals.
inline size_t ffma_noncausal_backward(int BH, int N, int D, int M, int num_sms) {
    const int spans = ffma_span_count(BH, N, D, M, num_sms);
    return 2 * sizeof(float) * (static_cast<size_t>(BH) * spans + BH) * state_words(D, M);
}

// Softmax KV-cache decode: positions of a head cut into ranges so that the grid
// is about eight waves of eight 256-thread CTAs per SM, at least 256 positions a range.
inline void softmax_decode_split(int BH, int total, int num_sms, int* splits, int* split_len) {
    int s = (64 * num_sms + std::max(BH, 1) - 1) / std::max(BH, 1);
    s = std::max(1, std::min(s, (total + 255) / 256));
    *split_len = (total + s - 1) / s;
    *splits = (total + *split_len - 1) / *split_len;
}

// Its per-range partials: running maximum, weight sum and D weighted-value sums.
inline size_t softmax_decode_scratch(int BH, int total, int D, int num_sms) {
    int splits = 1, len = 1;
    softmax_decode_split(BH, total, num_sms, &splits, &len);
    return sizeof(float) * static_cast<size_t>(BH) * splits * (D + 2);
}

// CUDA-core retention forward: per-span aggregates (D x M, no normaliser) and
// per-span total log2 decays, only when a head has several spans.
inline size_t ffma_retention_forward(int BH, int N, int D, int M, int num_sms) {
    const int spans = ffma_span_count(BH, N, D, M, num_sms);
    return spans > 1 ? sizeof(float) * static_cast<size_t>(BH) * spans * (static_cast<size_t>(D) * M + 1)
                     : 0;
}

// Degree-2 polynomial feature map (D = 32): the D (D + 1) / 2 = 528 features
// split into kPolySlices slices; a grid of heads x spans x slices of about two
// waves of one CTA per SM.
constexpr int kPolySlices = 3;
constexpr int kPolyFeatures = 32 * 33 / 2;
constexpr int kPolyChunk = 64;
inline void poly_spans(int BH, int N, int num_sms, int* spans, int* span_len) {
    const int chunks = (N + kPolyChunk - 1) / kPolyChunk;
    int s = (2 * num_sms + kPolySlices * std::max(BH, 1) - 1) / (kPolySlices * std::max(BH, 1));
    s = std::max(1, std::min(s, std::max(chunks, 1)));
    const int per = (chunks + s - 1) / s;
    *span_len = std::max(per, 1) * kPolyChunk;
    *spans = std::max(1, (N + *span_len - 1) / *span_len);
}
// The span aggregates of every slice ([BH][spans][features][M + 1]) and the
// fp32 numerator and denominator accumulator [BH][N][M + 1].
inline size_t poly2_scratch(int BH, int N, int M, int num_sms) {
    int spans = 1, len = 1;
    poly_spans(BH, N, num_sms, &spans, &len);
    const size_t agg = sizeof(float) * static_cast<size_t>(BH) * spans * kPolyFeatures * (M + 1);
    return up256(agg) + sizeof(float) * static_cast<size_t>(BH) * N * (M + 1);
}

// Tensor-core degree-2 map (bf16, D = 32, M = 64): four CTAs per head, each
// owning two 128-feature slices of the D^2 = 1024 features; the only scratch is
// the fp32 [numerator | normaliser | 15 copies] accumulator [BH][N][M + 16].
constexpr int kPolyTcGroups = 4;
inline size_t poly2_tc_scratch(int BH, int N) {
    return sizeof(float) * static_cast<size_t>(BH) * N * (64 + 16);
}

// Tensor-core causal kernels: the chunks of all heads cut into equal ranges,
// one per resident CTA (see tc_common.cuh, split_chunks).
inline int tc_units(int BH, int chunks_per_head, int slots) {
    const long long total = static_cast<long long>(BH) * chunks_per_head;
    const long long per = std::max(1LL, (total + slots - 1) / std::max(1, slots));
    return static_cast<int>((total + per - 1) / per);
}

}  // namespace plan
}  // namespace la
