// tc_common.cuh -- pieces shared by the tensor-core linear-attention kernels:
// chunk geometry, status bits, the phi transform of swizzled bf16 tiles,
// swizzled row stores, release/acquire flags and the TMA tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "tc_ptx.cuh"

namespace la {
namespace tcf {

using bf16 = __nv_bfloat16;
using namespace la::tc;

constexpr int L = 128;                      // chunk length = MMA M
constexpr int kThreads = 128;               // one thread per TMEM lane / tile row
constexpr uint32_t kAtom = 16384;           // one 128-row atom column (128 x 128 B)
constexpr uint32_t kWaitLimit = 1u << 24;   // mbarrier polls before giving up
constexpr uint32_t kSpinLimit = 1u << 22;   // flag polls (256 ns apart) before giving up

// Status bits written to the device error word.
constexpr unsigned kErrWait = 1u;      // a TMA or MMA completion never arrived
constexpr unsigned kErrLookback = 2u;  // an earlier span never published its state
constexpr unsigned kErrAlign = 4u;     // dynamic shared memory not 1024-byte aligned

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// 2^x on the special-function unit (ex2.approx, flush-to-zero).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// phi(x) = elu(x) + 1 written without a branch: max(x, 0) + e^min(x, 0), with
// e^u = 2^(u log2 e).  For x > 0 this is x + 1, for x <= 0 it is e^x.  The
// approximate 2^u is far more accurate than the 2^-9 rounding of bf16.
__device__ __forceinline__ float phi_fast(float x) {
    return fmaxf(x, 0.f) + ex2_approx(fminf(x, 0.f) * 1.4426950408889634f);
}

// phi on two packed bf16 values in packed bf16 arithmetic: max(x, 0) +
// 2^(min(x, 0) * log2 e), one exponential per pair.  For x > 0 the exponent
// is 0 and the sum is x + 1 rounded once; for x <= 0 it is e^x.  The product
// and the approximate 2^u are each within about one bf16 rounding, the size
// of the rounding the result gets anyway when stored as bf16.
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t x) {
    uint32_t r;
    asm("{\n\t.reg .b32 n, p, y, e;\n\t"
        "min.bf16x2 n, %1, %2;\n\t"
        "max.bf16x2 p, %1, %2;\n\t"
        "fma.rn.bf16x2 y, n, %3, %2;\n\t"
        "ex2.approx.ftz.bf16x2 e, y;\n\t"
        "fma.rn.bf16x2 %0, p, %4, e;\n\t}"
        : "=r"(r)
        : "r"(x), "r"(0u), "r"(0x3FB93FB9u), "r"(0x3F803F80u));  // 0, log2 e, 1 (bf16 pairs)
    return r;
}

// phi in place over `atoms` swizzled atom columns (1024 16-byte chunks each);
// rows >= valid become 0 when ZERO_TAIL (padding keys must not enter S or Z:
// phi(0) = 1).  Each thread works on 8 independent chunks at a time so that
// the loads, the exponentials and the stores of different chunks overlap.
template <bool ZERO_TAIL, int NT = kThreads>
__device__ __forceinline__ void phi_tile(uint8_t* tile, int atoms, int valid) {
    constexpr int U = 1024 / NT < 8 ? 1024 / NT : 8;  // chunks per thread per batch
    const int n = atoms * 1024;
    for (int base = threadIdx.x; base < n; base += NT * U) {
        uint4 u[U];
#pragma unroll
        for (int j = 0; j < U; ++j)
            u[j] = *reinterpret_cast<const uint4*>(tile + static_cast<size_t>(base + j * NT) * 16);
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int row = ((base + j * NT) & 1023) >> 3;
            if (ZERO_TAIL && row >= valid) {
                u[j] = make_uint4(0u, 0u, 0u, 0u);
            } else {
                u[j].x = phi_bf16x2(u[j].x);
                u[j].y = phi_bf16x2(u[j].y);
                u[j].z = phi_bf16x2(u[j].z);
                u[j].w = phi_bf16x2(u[j].w);
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j)
            *reinterpret_cast<uint4*>(tile + static_cast<size_t>(base + j * NT) * 16) = u[j];
    }
}

// phi of one Q atom and one K atom (K's rows >= valid become 0), worked by NT
// threads numbered `tid` = 0 .. NT - 1.  Each thread takes 1024 / NT chunks of
// each atom in one unguarded batch, all loads first, so that the loads, the
// exponentials and the stores overlap; the 1024 % NT chunks left over go one
// per thread.  (A loop of guarded batches, the form for any NT, ran 2.6 times
// slower at NT = 96.)
template <int NT>
__device__ __forceinline__ void phi_pair(uint8_t* tq, uint8_t* tk, int valid, int tid) {
    constexpr int U = 1024 / NT, TAIL = 1024 - NT * U;
    static_assert(U >= 1 && U <= 16, "chunks per thread");
    uint4 a[U], b[U];
#pragma unroll
    for (int j = 0; j < U; ++j) a[j] = *reinterpret_cast<const uint4*>(tq + (tid + j * NT) * 16);
#pragma unroll
    for (int j = 0; j < U; ++j) b[j] = *reinterpret_cast<const uint4*>(tk + (tid + j * NT) * 16);
#pragma unroll
    for (int j = 0; j < U; ++j) {
        a[j].x = phi_bf16x2(a[j].x);
        a[j].y = phi_bf16x2(a[j].y);
        a[j].z = phi_bf16x2(a[j].z);
        a[j].w = phi_bf16x2(a[j].w);
    }
#pragma unroll
    for (int j = 0; j < U; ++j) *reinterpret_cast<uint4*>(tq + (tid + j * NT) * 16) = a[j];
#pragma unroll
    for (int j = 0; j < U; ++j) {
        if (((tid + j * NT) >> 3) >= valid) {
            b[j] = make_uint4(0u, 0u, 0u, 0u);
        } else {
            b[j].x = phi_bf16x2(b[j].x);
            b[j].y = phi_bf16x2(b[j].y);
            b[j].z = phi_bf16x2(b[j].z);
            b[j].w = phi_bf16x2(b[j].w);
        }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) *reinterpret_cast<uint4*>(tk + (tid + j * NT) * 16) = b[j];
    if (TAIL > 0 && tid < TAIL) {
        const int c = NT * U + tid;
        uint4 x = *reinterpret_cast<const uint4*>(tq + c * 16);
        uint4 y = *reinterpret_cast<const uint4*>(tk + c * 16);
        x.x = phi_bf16x2(x.x);
        x.y = phi_bf16x2(x.y);
        x.z = phi_bf16x2(x.z);
        x.w = phi_bf16x2(x.w);
        if ((c >> 3) >= valid) {
            y = make_uint4(0u, 0u, 0u, 0u);
        } else {
            y.x = phi_bf16x2(y.x);
            y.y = phi_bf16x2(y.y);
            y.z = phi_bf16x2(y.z);
            y.w = phi_bf16x2(y.w);
        }
        *reinterpret_cast<uint4*>(tq + c * 16) = x;
        *reinterpret_cast<uint4*>(tk + c * 16) = y;
    }
}

// Stores 32 consecutive bf16 values (packed in pk[16]) of `row`, starting at
// column j0, into a K-major 128-row swizzled tile.
__device__ __forceinline__ void store_row32(uint8_t* tile, uint32_t atom_bytes, int row, int j0,
                                            const uint32_t (&pk)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int c = (j0 >> 3) + q;  // logical 16-byte chunk along the row
        *reinterpret_cast<uint4*>(tile + (c >> 3) * atom_bytes + swz(row, c & 7)) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
}

// ------------------------------------------------------------------ host

// Checkpoint slots per head (see kCkptChunks).
__host__ __device__ constexpr int ckpt_slots(int chunks_per_head) {
    return (chunks_per_head + kCkptChunks - 1) / kCkptChunks;
}

// Work split of the causal kernels: the chunks of all heads, head-major, cut
// into `units` equal ranges of `per` chunks, one per resident CTA (one wave,
// every CTA busy for the same number of chunks whatever the head count).
struct ChunkSplit {
    int per, units;
};
inline ChunkSplit split_chunks(int BH, int chunks_per_head, int slots) {
    const long long total = static_cast<long long>(BH) * chunks_per_head;
    const long long per = std::max(1LL, (total + slots - 1) / std::max(1, slots));
    return {static_cast<int>(per), static_cast<int>((total + per - 1) / per)};
}

// One unit's range [start, end) of global chunk indices (head h = index / CH)
// and how it meets its neighbours.  Its pieces in successive heads are its
// segments: only the first can continue a head begun by earlier units, and
// only the last can stop inside a head that later units continue.
struct UnitRange {
    int start, end;  // global chunk indices
    int hA, hB;      // heads of the first and the last segment
    bool look;       // the first segment continues a head: earlier units hold its prefix
    bool publish;    // the last segment stops inside its head: later units need its sum
    int u_first;     // first unit holding a chunk of head hA
    int u_last;      // last unit holding a chunk of head hB
    __device__ UnitRange(int u, int per, int CH, int BH) {
        const int total = BH * CH;
        start = u * per;
        end = min(total, start + per);
        hA = start / CH;
        hB = (end - 1) / CH;
        look = start != hA * CH;
        publish = end != (hB + 1) * CH;
        u_first = hA * CH / per;
        u_last = ((hB + 1) * CH - 1) / per;
    }
};

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(f);
    });
    return fn;
}

// 3-D map over a [BH][N][C] bf16 tensor with a {64, 128, 1} box and the
// 128-byte swizzle; rows past N read as zero and are not written.
inline cudaError_t make_map(CUtensorMap* m, const void* base, int BH, int N, int C) {
    EncodeTiled enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2, static_cast<cuuint64_t>(N) * C * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(L), 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D map over a [BH][N][C] fp32 tensor with a {32, rows, 1} box (128 bytes of
// a row per box) and the 128-byte swizzle.
inline cudaError_t make_map_f32(CUtensorMap* m, const void* base, int BH, int N, int C, int rows = L) {
    EncodeTiled enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(N),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 4, static_cast<cuuint64_t>(N) * C * 4};
    cuuint32_t box[3] = {32, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tcf
}  // namespace la
